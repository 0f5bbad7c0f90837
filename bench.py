#!/usr/bin/env python
"""Benchmark of the continuous-batching paged step on GB300.

One step = one pass of the hot path over one packed batch: kv_append of the step's new
K/V rows into the 16-token block pool, then paged_attention_step (metadata prep,
tcgen05 prefill tiles beside the split-KV decode, then the combine of split rows), all
through the C ABI.

Metric: packed query tokens/s per attention layer (T / step time), and the decode
kernel's KV-read GB/s against the measured HBM peak.  Default workload: the largest
single-GPU step, chunked prefill under an 8192-token budget (four 2048-token chunks
after 0/2048/4096/6144 cached tokens plus 32 decode rows with context ~ U[512, 8192],
GQA 32/8, d 128, bf16, 32768-block pool); its roofline is the prefill kernel's dense
bf16 fraction.  The same JSON line carries the decode-heavy step (256 decode rows,
lognormal contexts: the decode kernel's HBM fraction) and the mixed step (64 decode
rows + two 512-token chunks), each timed the same way, under "workloads".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config chunked|mixed|decode|tiny|trace]
  python bench.py --impl reference ...   # the CPU oracle on the same workload

Under torchrun (N > 1) every rank runs its own replica of the step on its own GPU (the
requests of different replicas are independent: weak scaling, no collective on the
data path); rank 0 prints one JSON line with the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# The CPU oracle runs one process per host core, each with BLAS on one thread (set
# before numpy loads; spawned workers import this module again and inherit it).
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

METRIC = "packed query tokens/s per attention layer; decode KV-read GB/s vs GB300 HBM peak"
UNIT = "tokens/s"
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0
L2_FLUSH_BYTES = 256 << 20
CSRC = os.path.join(ROOT, "continuous_batching_paged_step_gb300", "csrc")
# the files a kernel's code lives in (its .cu, the device-code header it shares with the
# mixed step kernel, the common device helpers): a change to any of them makes recorded
# ncu counters stale
KERNEL_SOURCES = {"decode_splitkv": ("attn_decode.cu", "attn_decode.cuh", "kvp_device.cuh"),
                  "splitkv_combine": ("attn_decode.cu", "attn_decode.cuh", "kvp_device.cuh"),
                  "prefill_tcgen05": ("attn_prefill.cu", "attn_prefill.cuh", "kvp_device.cuh"),
                  "kv_append": ("kv_append.cu", "kvp_device.cuh"), "step_prep": ("attn_prep.cu", "kvp_device.cuh")}


# ------------------------------------------------------------------ workload algebra

def work_of(spec):
    """Algorithmic work of one step (what the method must touch, not what a kernel does)."""
    dec_bytes = 0
    pairs = 0
    for q, c in zip(spec.q_lens, spec.ctx_lens):
        if q == 1:
            n = c + 1
            # K+V of every visible key (8 heads x 128 x bf16 x 2), Q and O rows, table entries
            dec_bytes += n * 4096 + 8192 + 8192 + 4 * (-(-n // 16))
        elif q > 1:
            pairs += q * c + q * (q + 1) // 2       # visible (query, key) pairs
    T = spec.num_tokens
    return {
        "decode_bytes": dec_bytes,
        # QK^T and P.V over visible pairs: 2 x 2 x 128 FLOPs per pair per query head
        "prefill_flops": pairs * 32 * 2 * 2 * 128,
        # kv_append reads T new K/V rows and writes them into the pool
        "append_bytes": T * 2048 * 2 * 2,
    }


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), \
            "measured (MEASURED_PEAKS.json)"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def source_sha(kernel):
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on this source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = source_sha(kernel)
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            kv = dict(tok.split("=", 1) for tok in line.split() if "=" in tok)
            if kv.get("kernel") == kernel and kv.get("workload") == workload and kv.get("src_sha") == sha:
                return float(kv["bytes_per_launch"])
    return None


# ------------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[6 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[4]) for r in rows if r[4].replace(".", "").isdigit())
                if any(r[4].replace(".", "").isdigit() for r in rows) else None}


# --------------------------------------------------------------------- oracle leg

def oracle_sample_rows(T, n_rows, shift=0):
    """n_rows packed rows evenly spaced over the whole step (every row when n_rows >= T), so
    decode rows and prefill rows at every position enter in proportion and the oracle's
    rows/s stands for the whole step's.  Sample `shift` starts at a golden-ratio fraction of
    the spacing, so that successive samples cover all rows."""
    n = max(1, min(T, int(n_rows)))
    frac = (shift * 0.6180339887498949) % 1.0
    return np.unique(np.minimum(((np.arange(n) + frac) * (T / n)).astype(np.int64), T - 1))


_WORKER_INPUTS = {}


def _oracle_inputs(config):
    """The step's inputs from the seeded generator, drawn once per process."""
    if config not in _WORKER_INPUTS:
        from continuous_batching_paged_step_gb300 import workloads as wl
        _WORKER_INPUTS[config] = wl.make_inputs(wl.CONFIGS[config]())
    return _WORKER_INPUTS[config]


def _oracle_worker_init(config):
    _oracle_inputs(config)


def _oracle_worker_ping(_):
    time.sleep(0.05)
    return os.getpid()


def _oracle_worker_rows(args):
    config, rows = args
    import oracle
    inp = _oracle_inputs(config)
    out = oracle.step_reference(inp, rows=rows)
    assert np.isfinite(out[rows]).all()
    return len(rows)


def oracle_tasks(cu_seqlens_q, context_lens, rows, n_tasks):
    """Cut a sample of packed rows into about n_tasks lists, each holding rows of one
    request of about equal oracle cost (a row scores its position + 1 keys), longest
    first: the order a pool of workers takes them in."""
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    ctx = np.asarray(context_lens, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    req = np.searchsorted(cu, rows, side="right") - 1
    cost = ctx[req] + (rows - cu[req]) + 1
    target = max(float(cost.sum()) / max(1, n_tasks), float(cost.max()))
    tasks = []
    for r in np.unique(req):
        sel = req == r
        cur, acc = [], 0.0
        for x, c in zip(rows[sel], cost[sel]):
            if cur and acc + c > target:
                tasks.append((acc, cur))
                cur, acc = [], 0.0
            cur.append(int(x))
            acc += float(c)
        if cur:
            tasks.append((acc, cur))
    tasks.sort(key=lambda t: -t[0])
    return [t[1] for t in tasks]


class OracleTimer:
    """The oracle as it stands, timed on the host's cores: `workers` processes (spawned,
    so safe to start after CUDA is initialised), each with BLAS on one thread and its own
    copy of the step's inputs drawn before any timing; a sample of rows is cut into
    per-request tasks that the workers take longest first, and the wall time of the whole
    sample is measured.  workers = 1 runs in this process."""

    def __init__(self, config, workers=None):
        from continuous_batching_paged_step_gb300 import workloads as wl
        self.config = config
        spec = wl.CONFIGS[config]()
        self.cu = np.zeros(spec.num_reqs + 1, dtype=np.int64)
        self.cu[1:] = np.cumsum(spec.q_lens)
        self.ctx = np.asarray(spec.ctx_lens, dtype=np.int64)
        self.workers = max(1, int(workers if workers else (os.cpu_count() or 1)))
        self.pool = None
        if self.workers > 1:
            self.pool = mp.get_context("spawn").Pool(self.workers, initializer=_oracle_worker_init,
                                                     initargs=(config,))
            seen = set()
            for _ in range(50):    # every worker has drawn its inputs once it answers
                seen.update(self.pool.map(_oracle_worker_ping, range(4 * self.workers), chunksize=1))
                if len(seen) >= self.workers:
                    break
        else:
            _oracle_inputs(config)

    def time_rows(self, rows):
        """(rows computed, wall seconds) for one sample."""
        if self.pool is None:
            t0 = time.perf_counter()
            n = _oracle_worker_rows((self.config, [int(x) for x in rows]))
            return n, time.perf_counter() - t0
        tasks = oracle_tasks(self.cu, self.ctx, rows, self.workers)
        t0 = time.perf_counter()
        n = sum(self.pool.map(_oracle_worker_rows, [(self.config, t) for t in tasks], chunksize=1))
        return n, time.perf_counter() - t0

    def close(self):
        if self.pool is not None:
            self.pool.close()
            self.pool.join()
            self.pool = None


def time_oracle(config, n_rows, min_seconds=0.0, shift=0, timer=None):
    """Wall time of the oracle over a sample of n_rows rows of the step, repeated (each
    pass shifted) until at least `min_seconds` have been timed.  Returns (rows computed,
    wall seconds, passes).  Input generation is outside the timed calls."""
    own = timer is None
    timer = timer or OracleTimer(config, workers=1)
    from continuous_batching_paged_step_gb300 import workloads as wl
    T = wl.CONFIGS[config]().num_tokens
    n, wall, passes = 0, 0.0, 0
    try:
        while passes == 0 or wall < min_seconds:
            rows = oracle_sample_rows(T, n_rows, shift + passes)
            k, w = timer.time_rows(rows)
            n += k
            wall += w
            passes += 1
    finally:
        if own:
            timer.close()
    return n, wall, passes


# ---------------------------------------------------------------------- GPU arm

SIDE_WORKLOADS = ("decode", "mixed", "chunked")


def rooflines(spec, kern):
    """(dominant kernel's roofline, the other attention kernel's) for one workload."""
    hbm, bf16, _, peak_src = peaks()
    work = work_of(spec)
    dec_us = kern.get("decode_splitkv", {}).get("avg_us")
    pre_us = kern.get("prefill_tcgen05", {}).get("avg_us")
    dominant = max(kern, key=lambda k: kern[k]["avg_us"] * kern[k]["launches"]) if kern else None
    rl_decode = None
    if dec_us:
        ach = work["decode_bytes"] / (dec_us * 1e-6) / 1e9
        rl_decode = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(ach / hbm, 4), "traffic": ncu_traffic("decode_splitkv", spec.name),
                     "kernel": "decode_splitkv", "algorithmic_bytes_per_launch": work["decode_bytes"],
                     "avg_us": round(dec_us, 2), "peak_source": f"hbm_gbs, {peak_src}"}
    rl_prefill = None
    if pre_us and work["prefill_flops"]:
        ach = work["prefill_flops"] / (pre_us * 1e-6) / 1e12
        rl_prefill = {"bound": "tensor", "achieved": round(ach, 1), "peak": bf16, "unit": "TFLOP/s",
                      "frac": round(ach / bf16, 4), "traffic": ncu_traffic("prefill_tcgen05", spec.name),
                      "kernel": "prefill_tcgen05", "algorithmic_flops_per_launch": work["prefill_flops"],
                      "avg_us": round(pre_us, 2), "peak_source": f"bf16_tflops (burst), {peak_src}"}
    roofline = rl_prefill if dominant == "prefill_tcgen05" else rl_decode
    secondary = rl_decode if roofline is rl_prefill else rl_prefill
    return roofline, secondary


def measure_step(spec, a, dev, dist, world, flush, with_e2e):
    """One workload on this GPU: W warm-up steps, K timed steps (CUDA events on the
    launching stream, L2 flushed between steps outside the events), K more steps with the
    library's events around each of its kernels (per-kernel durations), and optionally
    the end-to-end leg.  Returns the measurements; closes the step."""
    import torch
    from continuous_batching_paged_step_gb300 import kvpaged as kp
    from continuous_batching_paged_step_gb300 import replicas, runner, workloads as wl
    inp = wl.make_inputs(spec)
    step = runner.PagedStep(inp, device=dev)
    stream = torch.cuda.current_stream(dev)
    try:
        for i in range(a.warmup):
            flush.fill_(i & 0xFF)
            step.run()
        torch.cuda.synchronize(dev)
        st = step.error()
        if st != (0, 0):
            raise RuntimeError(f"{spec.name}: device error word after warm-up: {st}")

        def timed_steps(n):
            starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
            ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
            replicas.barrier(dist)
            torch.cuda.synchronize(dev)
            for i in range(n):
                flush.fill_((i + 1) & 0xFF)        # L2 flush between steps, outside the step's events
                starts[i].record(stream)
                step.run()
                ends[i].record(stream)
            torch.cuda.synchronize(dev)
            replicas.barrier(dist)
            return [s_.elapsed_time(e) for s_, e in zip(starts, ends)]

        # the steps as a user runs them (no timing events inside the library calls)
        launches0 = kp.kv_pool_launch_count(step.pool.handle)
        wall0 = time.perf_counter()
        step_ms = timed_steps(a.steps)
        wall = time.perf_counter() - wall0
        launches = kp.kv_pool_launch_count(step.pool.handle) - launches0
        # the same number of steps with CUDA events around every kernel the library
        # launches, on its launch stream: per-kernel durations for the roofline
        kp.kv_pool_enable_timing(step.pool.handle, 8 * a.steps + 16)
        step_ms_kernels = timed_steps(a.steps)
        per_kernel = kp.kv_pool_read_timing(step.pool.handle)
        kp.kv_pool_enable_timing(step.pool.handle, 0)
        st = step.error()
        if st != (0, 0):
            raise RuntimeError(f"{spec.name}: device error word after the timed steps: {st}")
        total_ms = replicas.max_over_ranks(dist, sum(step_ms), device=dev)
        e2e = run_e2e(a, step, stream, dev, dist, world, total_ms / a.steps) if with_e2e else None
    finally:
        step.close()
    kern = {name: {"launches": n, "avg_us": 1e3 * ms / n} for name, (n, ms) in per_kernel.items() if n}
    T = spec.num_tokens
    return {"value": replicas.aggregate_rate(T * a.steps, world, total_ms), "total_ms": total_ms,
            "ms_per_step_with_kernel_events": sum(step_ms_kernels) / a.steps, "kern": kern,
            "launches": int(launches), "wall": wall, "e2e": e2e}


def run_gpu(a):
    import torch
    from continuous_batching_paged_step_gb300 import build as b
    b.build()
    from continuous_batching_paged_step_gb300 import replicas, workloads as wl
    rank, world, local = replicas.dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = replicas.init("nccl", device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    spec = wl.CONFIGS[a.config]()
    sides = [] if (a.no_side_workloads or a.config not in SIDE_WORKLOADS) else \
        [c for c in SIDE_WORKLOADS if c != a.config]
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.25)
    main = measure_step(spec, a, dev, dist, world, flush, with_e2e=True)
    side = {}
    for c in sides:
        sp = wl.CONFIGS[c]()
        side[sp.name] = (sp, measure_step(sp, a, dev, dist, world, flush, with_e2e=False))
    clk = clocks.stop()
    del flush
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return None

    roofline, secondary = rooflines(spec, main["kern"])
    workloads = {}
    for name, (sp, m) in side.items():
        rl, rl2 = rooflines(sp, m["kern"])
        workloads[name] = {"value": round(m["value"], 1), "unit": UNIT, "steps": a.steps,
                           "ms_per_step": round(m["total_ms"] / a.steps, 5), "num_tokens": sp.num_tokens,
                           "roofline": rl, "roofline_secondary": rl2,
                           "kernels_us": {k: round(v["avg_us"], 2) for k, v in m["kern"].items()},
                           "gpu_launches": m["launches"]}

    def frac_of(rl_pair, kernel):
        for rl in rl_pair:
            if rl and rl["kernel"] == kernel:
                return rl["frac"]
        return None

    targets = {"prefill_tensor_frac": frac_of((roofline, secondary), "prefill_tcgen05"),
               "prefill_tensor_frac_workload": spec.name}
    dh = wl.CONFIGS["decode"]().name
    if dh == spec.name:
        targets["decode_heavy_hbm_frac"] = frac_of((roofline, secondary), "decode_splitkv")
    elif dh in workloads:
        targets["decode_heavy_hbm_frac"] = frac_of((workloads[dh]["roofline"], workloads[dh]["roofline_secondary"]),
                                                   "decode_splitkv")
    targets["targets"] = "decode-dominated steps >= 0.70 of HBM peak; prefill tiles >= 0.50 of dense bf16 peak"

    cpu = None
    if not a.no_cpu_baseline:
        cpu = cpu_baseline(a, spec)

    line = {
        "metric": METRIC, "value": round(main["value"], 1), "unit": UNIT, "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": round(main["total_ms"] / a.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": step_config(spec, world),
        "decode_kv_gbs": next((rl["achieved"] for rl in (roofline, secondary) if rl and rl["kernel"] == "decode_splitkv"),
                              None),
        "roofline": roofline, "roofline_secondary": secondary, **targets,
        "kernels_us": {k: round(v["avg_us"], 2) for k, v in main["kern"].items()},
        "ms_per_step_with_kernel_events": round(main["ms_per_step_with_kernel_events"], 5),
        "workloads": workloads,
        "cpu_baseline": cpu, "e2e": main["e2e"], "clocks": clk, "gpu_launches": main["launches"],
        "wall_s_timed": round(main["wall"], 3),
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return line


def cpu_baseline(a, spec):
    """The oracle on the host's cores, on a bounded sample of the workload: a short probe
    sizes one pass (as many evenly spaced rows as about --oracle-seconds allow, the whole
    step when it fits), repeated until that much oracle time is measured."""
    timer = OracleTimer(a.config, workers=a.oracle_workers or None)
    try:
        T = spec.num_tokens
        n_probe, w_probe, _ = time_oracle(a.config, 4 * timer.workers, timer=timer)
        n_pass = min(T, max(4 * timer.workers, int(n_probe / max(w_probe, 1e-6) * a.oracle_seconds)))
        n_rows, owall, passes = time_oracle(a.config, n_pass, a.oracle_seconds, timer=timer)
    finally:
        timer.close()
    return {"value": round(n_rows / owall, 3), "unit": UNIT, "cores": timer.workers, "kind": "oracle",
            "sample": f"{passes} pass(es) over {n_rows // passes} of {T} packed rows of the {spec.name} step, "
                      f"evenly spaced over the step (decode and prefill rows in proportion), fp64 numpy, "
                      f"{timer.workers} processes with one BLAS thread each, {owall:.1f} s"}


E2E_MIN_MS = 200.0
E2E_MAX_STEPS = 5000


def run_e2e(a, step, stream, dev, dist, world, est_ms):
    """Same metric through the C ABI with host buffers, as a serving loop runs it: every
    step's inputs go host -> device from pinned memory and its output device -> host,
    inside the timed region.  The copies are pipelined with the compute: two sets of
    device inputs/outputs, uploads on one stream, downloads on another, so step i+1's
    upload and step i-1's download overlap step i's kernels (and each other: an upload
    waits only for the step that last read its input set, a step only for the download of
    the output set it overwrites).  No L2 flush here: every step streams the decode rows'
    whole KV history (hundreds of MB, more than L2).  At least --steps steps are timed, and
    enough that the timed region lasts about E2E_MIN_MS (the pipeline's fill and drain are
    then a small part of it); the count is reported."""
    import torch
    from continuous_batching_paged_step_gb300 import kvpaged as kp
    from continuous_batching_paged_step_gb300 import replicas
    inp = step.inp
    names = ("q", "k_new", "v_new", "cu_seqlens_q", "context_lens", "block_tables")
    # the step's inputs packed into one pinned host blob (each at a 256-byte offset), so that
    # a step's upload is one copy; the device sets hold the same layout, viewed per input
    offs, total_bytes = {}, 0
    for nm in names:
        t = getattr(step, nm)
        offs[nm] = total_bytes
        total_bytes += (t.numel() * t.element_size() + 255) & ~255

    def views(blob):
        out = {}
        for nm in names:
            t = getattr(step, nm)
            nb = t.numel() * t.element_size()
            out[nm] = blob[offs[nm]:offs[nm] + nb].view(t.dtype).view(t.shape)
        return out

    host_blob = torch.empty(total_bytes, dtype=torch.uint8).pin_memory()
    for nm, v in views(host_blob).items():
        v.copy_(getattr(step, nm).cpu())
    dev_blobs = [torch.empty(total_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    bufs = [views(b) for b in dev_blobs]
    out_h = [torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory() for _ in range(2)]
    outs = [torch.empty_like(step.out) for _ in range(2)]
    h2d = total_bytes
    d2h = out_h[0].numel() * out_h[0].element_size()
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    n = int(min(E2E_MAX_STEPS, max(a.steps, math.ceil(E2E_MIN_MS / max(est_ms, 1e-3)))))
    # events reused by parity: step i waits on those step i - 2 recorded, before it records its own
    loaded = torch.cuda.Event()
    computed = [torch.cuda.Event() for _ in range(2)]   # step's kernels finished (its input set is free)
    done = [torch.cuda.Event() for _ in range(2)]       # step's output is on the host

    def run(count, timed):
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        if timed:
            t0.record(up)
        for i in range(count):
            j = i % 2
            b = bufs[j]
            if i >= 2:
                up.wait_event(computed[j])          # step i-2 no longer reads this input set
            with torch.cuda.stream(up):
                dev_blobs[j].copy_(host_blob, non_blocking=True)
                loaded.record(up)
            stream.wait_event(loaded)
            if i >= 2:
                stream.wait_event(done[j])          # step i-2's output left this output set
            kp.kv_append(step.pool.handle, b["k_new"], b["v_new"], b["cu_seqlens_q"], b["context_lens"],
                         b["block_tables"], stream=stream)
            kp.paged_attention_step(step.pool.handle, b["q"], outs[j], b["cu_seqlens_q"], b["context_lens"],
                                    b["block_tables"], step.max_q_len, step.max_context_len, step.softmax_scale,
                                    step.workspace, stream=stream)
            computed[j].record(stream)
            down.wait_event(computed[j])
            with torch.cuda.stream(down):
                out_h[j].copy_(outs[j], non_blocking=True)
                done[j].record(down)
        if timed:
            t1.record(down)
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1) if timed else 0.0

    run(4, False)
    total = replicas.max_over_ranks(dist, run(n, True), device=dev)
    T = inp.spec.num_tokens
    return {"value": round(replicas.aggregate_rate(T * n, world, total), 1), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": n,
            "pipelining": "double-buffered device inputs/outputs, each step's inputs one packed upload; "
                          "uploads, kernels and downloads on three streams"}


# ---------------------------------------------------------------- reference arm

def step_config(spec, world):
    """The `config` object of a step workload's JSON line (both arms)."""
    return {"workload": spec.name, "num_tokens": spec.num_tokens, "num_reqs": spec.num_reqs,
            "decode_rows": sum(1 for q in spec.q_lens if q == 1),
            "prefill_chunks": [[q, c] for q, c in zip(spec.q_lens, spec.ctx_lens) if q > 1],
            "heads": "32 q / 8 kv, d 128", "block_size": 16, "kv_pool_blocks": spec.num_blocks,
            "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write outside the step events)",
            "parallelism": f"replicas x{world}"}


def run_reference(a):
    """The CPU oracle as it stands, on the same workload, on the host's cores: each step is
    the oracle over a bounded sample of the step's rows, sized so the whole run takes a
    few minutes."""
    if int(os.environ.get("RANK", "0")) != 0:
        return None
    from continuous_batching_paged_step_gb300 import workloads as wl
    spec = wl.CONFIGS[a.config]()
    timer = OracleTimer(a.config, workers=a.oracle_workers or None)
    budget_s = 150.0
    try:
        # a timed probe with a small sample sizes the per-step sample to the budget (at
        # least 8 evenly spaced rows a step)
        n_probe, w, _ = time_oracle(a.config, 4 * timer.workers, timer=timer)
        per_step_target = budget_s / max(1, a.steps + a.warmup)
        n_pass = min(spec.num_tokens, max(8, int(n_probe / max(w, 1e-6) * per_step_target)))
        rows_timed, t_timed = 0, 0.0
        for i in range(a.warmup + a.steps):
            n_rows, w, _ = time_oracle(a.config, n_pass, shift=i, timer=timer)
            if i >= a.warmup:
                rows_timed += n_rows
                t_timed += w
    finally:
        timer.close()
    per = t_timed / max(1, a.steps)
    value = rows_timed / max(t_timed, 1e-9)
    sample = (f"{n_pass} of {spec.num_tokens} packed rows per step of the {spec.name} step, evenly spaced over "
              f"the step (decode and prefill rows in proportion, shifted from step to step), {timer.workers} "
              f"processes with one BLAS thread each; value = rows / time over the timed steps")
    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(per * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": step_config(spec, int(os.environ.get("WORLD_SIZE", "1"))),
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": timer.workers, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return line


def run_trace(a):
    """The trace replay: 512 requests (Poisson arrivals, shared 1024-token system prompt in
    refcounted blocks, lognormal prompts and outputs), FCFS under an 8192-token budget, a
    40 GiB pool; every step is kv_append + paged_attention_step.  The trace is served once
    as the Python driver runs it (it plans each step and draws its inputs on the host,
    slower than the GPU step: those step windows are reported as `served`), recording
    every step's device inputs and block-manager calls; the headline value then serves the
    recorded steps again on a fresh pool, back to back, with the inputs resident in HBM
    (packed tokens over the GPU time of the whole replay).  A second replay with events
    around every kernel gives the per-kernel split."""
    import torch
    from continuous_batching_paged_step_gb300 import build as b
    b.build()
    from continuous_batching_paged_step_gb300 import kvpaged as kp
    from continuous_batching_paged_step_gb300 import workloads as wl
    from continuous_batching_paged_step_gb300.trace import TraceRunner
    ts = wl.TraceSpec()
    tr = TraceRunner(ts)
    w0 = time.perf_counter()
    tr.run(record=True)
    wall = time.perf_counter() - w0
    st = kp.kv_pool_get_error(tr.pool.handle)
    if st != (0, 0):
        raise RuntimeError(f"device error word after the trace: {st}")
    served = tr.summary()
    rep = tr.replay()
    rep_ev = tr.replay(timing_launches=8 * 4000)
    tr.close()
    per_kernel = rep_ev["kernels"]
    hbm, bf16, _, peak_src = peaks()
    n_dec, ms_dec = per_kernel["decode_splitkv"]
    dec_gbs = served["decode_bytes"] / (ms_dec / 1e3) / 1e9 if ms_dec else None
    line = {"metric": METRIC, "value": round(rep["tokens_per_s"], 1), "unit": UNIT, "n_gpus": 1, "steps": rep["steps"],
            "warmup": 0, "ms_per_step": round(rep["gpu_ms"] / max(1, rep["steps"]), 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": ts.name, "requests": ts.n_requests, "shared_prefix": ts.shared_prefix,
                       "budget": ts.budget, "kv_pool_blocks": ts.pool_blocks,
                       "arrivals_per_step": ts.arrivals_per_step,
                       "l2": "not flushed: consecutive steps back to back, as served",
                       "timed": "recorded steps replayed back to back (inputs in HBM, block-manager calls between steps)"},
            "replay": {k: (round(v, 4) if isinstance(v, float) else v) for k, v in rep.items()},
            "served": {k: (round(v, 4) if isinstance(v, float) else v) for k, v in served.items()},
            # decode GB/s counts every request's shared-prefix blocks once per read, as the
            # algorithm reads them; they are the same physical blocks (L2-resident), so this
            # may exceed the HBM rate
            "decode_kv_gbs": round(dec_gbs, 1) if dec_gbs else None,
            "kernels_ms_total": {k: round(v[1], 3) for k, v in per_kernel.items() if v[0]},
            "gpu_ms_with_kernel_events": round(rep_ev["gpu_ms"], 3),
            "kernel_busy_tokens_per_s": round(rep["tokens"] / (sum(v[1] for v in per_kernel.values()) / 1e3), 1),
            "wall_s": round(wall, 1)}
    print(json.dumps(line), flush=True)


def main():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", choices=["chunked", "mixed", "decode", "tiny", "trace"], default="chunked")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-side-workloads", action="store_true",
                   help="time only --config (by default the chunked, mixed and decode-heavy steps are all timed "
                        "and the others reported under 'workloads')")
    p.add_argument("--oracle-seconds", type=float, default=10.0,
                   help="the cpu_baseline repeats its sample until this much oracle time is measured")
    p.add_argument("--oracle-workers", type=int, default=0,
                   help="oracle processes for the CPU legs (0: one per host core)")
    a = p.parse_args()
    if a.warmup < 3:
        p.error("--warmup must be at least 3")
    if a.impl == "reference":
        run_reference(a)
    elif a.config == "trace":
        run_trace(a)
    else:
        run_gpu(a)


if __name__ == "__main__":
    main()
