"""Trace replay: a stream of requests served by iteration-level scheduling through the
paged step, one packed step per iteration.

Scheduling follows the pages' description of continuous batching:
* every iteration re-decides who runs (page "11.2 连续批处理与 PagedAttention", section
  11.2.2; page "Continuous Batching" on k4i.top, section "iteration-level scheduling"):
  finished requests leave and free their blocks, waiting requests are admitted FCFS;
* a per-step token budget is filled with all decode tokens first and the rest goes to
  prefill chunks (page "11.2", section 11.2.5, "分块 Prefill"); a long prompt is cut
  into chunks across steps (page "Continuous Batching 深入实现", section "第三层");
* KV memory is taken block by block as a request grows (page "11.2", section 11.2.3)
  and returned when it finishes;
* every request starts with the same system prompt, held once in full, read-only,
  refcounted blocks that all requests' block tables reference (page "11.2", sections
  11.2.3-11.2.4; page "连续批处理与 PagedAttention 原理", section "前缀共享").
A request's first output token comes with its last prefill chunk; each later token is
one decode row (page "Continuous Batching", section "与 KV cache 的关系").  Sampled
tokens are stood in for by seeded K/V rows; there is no model.

`Scheduler` is host-only (it takes allocator callbacks, so it runs on the C-ABI pool or
on anything with the same three calls).  `TraceRunner` drives the GPU step.
"""
from __future__ import annotations

import collections
import math
import time
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

from .workloads import BLOCK_SIZE, TraceRequest, TraceSpec, make_trace, trace_rows


@dataclass
class RunState:
    req: TraceRequest
    shared: int                        # tokens of the shared prefix (full blocks)
    state: str = "waiting"             # waiting | prefill | decode | done
    prefilled: int = 0                 # own prompt tokens in the cache
    fed: int = 0                       # decode tokens in the cache
    generated: int = 0                 # output tokens produced so far
    blocks: list = field(default_factory=list)   # own physical blocks, in table order
    chunks: list = field(default_factory=list)   # (first position, tokens) of every chunk fed
    admitted: int = -1
    finished: int = -1

    @property
    def cached(self) -> int:
        return self.shared + self.prefilled + self.fed


@dataclass
class StepPlan:
    step: int
    entries: list                      # (RunState, context_len, q_len) in packing order

    @property
    def num_tokens(self) -> int:
        return sum(q for _, _, q in self.entries)


class Scheduler:
    """FCFS iteration-level scheduler with a token budget, decode first."""

    def __init__(self, trace, ts: TraceSpec, shared_blocks, alloc, ref, free):
        if ts.shared_prefix % BLOCK_SIZE:
            raise ValueError("the shared prefix must be whole blocks (only full blocks are shared)")
        self.ts = ts
        self.trace = trace
        self.shared_blocks = list(shared_blocks)
        self._alloc, self._ref, self._free = alloc, ref, free
        self.waiting = collections.deque()
        self.running = []                  # admission order
        self.done = []
        self.next_arrival = 0
        self.step = 0

    def finished(self) -> bool:
        return self.next_arrival == len(self.trace) and not self.waiting and not self.running

    def _grow(self, rs: RunState, upto: int):
        """Own blocks so positions < upto are backed (on-demand growth)."""
        need = -(-(upto - rs.shared) // BLOCK_SIZE)
        if need > len(rs.blocks):
            rs.blocks.extend(int(b) for b in self._alloc(need - len(rs.blocks)))

    def plan(self) -> StepPlan:
        ts, step = self.ts, self.step
        while self.next_arrival < len(self.trace) and self.trace[self.next_arrival].arrival <= step:
            self.waiting.append(RunState(self.trace[self.next_arrival], ts.shared_prefix))
            self.next_arrival += 1
        budget = ts.budget
        entries = []
        for rs in self.running:                              # decode rows first
            if budget == 0:
                break
            if rs.state == "decode":
                entries.append((rs, rs.cached, 1))
                budget -= 1
        for rs in self.running:                              # continuing prefill chunks
            if budget == 0:
                break
            if rs.state == "prefill":
                c = min(rs.req.prompt_len - rs.prefilled, budget)
                entries.append((rs, rs.cached, c))
                budget -= c
        while self.waiting and budget > 0 and (ts.max_num_seqs == 0 or len(self.running) < ts.max_num_seqs):
            rs = self.waiting.popleft()                      # admit FCFS
            rs.state, rs.admitted = "prefill", step
            self._ref(self.shared_blocks)
            self.running.append(rs)
            c = min(rs.req.prompt_len, budget)
            entries.append((rs, rs.cached, c))
            budget -= c
        for rs, ctx, q in entries:
            self._grow(rs, ctx + q)
        return StepPlan(step, entries)

    def commit(self, plan: StepPlan):
        """Advance every scheduled request past the step that just ran."""
        for rs, ctx, q in plan.entries:
            rs.chunks.append((ctx, q))
            if rs.state == "prefill":
                rs.prefilled += q
                if rs.prefilled == rs.req.prompt_len:
                    rs.generated, rs.state = 1, "decode"     # first token with the last chunk
            else:
                rs.fed += 1
                rs.generated += 1
            if rs.generated >= rs.req.output_len:
                rs.state, rs.finished = "done", plan.step
                self._free(self.shared_blocks + rs.blocks)
                rs.blocks = []
        self.running = [rs for rs in self.running if rs.state != "done"]
        self.done.extend(rs for rs, _, _ in plan.entries if rs.state == "done" and rs.finished == plan.step)
        self.step += 1

    def table_row(self, rs: RunState, width: int) -> np.ndarray:
        row = np.full(width, -1, dtype=np.int32)
        ids = self.shared_blocks + rs.blocks
        row[:len(ids)] = ids
        return row


def static_batch_steps(lengths, batch: int):
    """Steps of static batching: waves of `batch` requests, each wave as long as its
    longest request (page "11.2", section 11.2.1)."""
    return sum(max(lengths[i:i + batch]) for i in range(0, len(lengths), batch))


def history(ts: TraceSpec, rs: RunState):
    """K and V rows (bf16 bits) of every position a request has in the cache, rebuilt from
    the seeded chunks: the shared prefix, then each chunk it fed."""
    parts_k, parts_v = [], []
    _, k, v = trace_rows(ts.seed, -1, 0, ts.shared_prefix)
    parts_k.append(k)
    parts_v.append(v)
    for start, n in rs.chunks:
        _, k, v = trace_rows(ts.seed, rs.req.rid, start, n)
        parts_k.append(k)
        parts_v.append(v)
    return np.concatenate(parts_k), np.concatenate(parts_v)


class TraceRunner:
    """Runs a trace on the GPU: every step is kv_append + paged_attention_step.

    `run(record=True)` also keeps every step's device inputs and the block-manager calls
    made around it, so that `replay()` can serve the same steps again, back to back, on a
    fresh pool: the scheduling and the input generation (host work, slower than the GPU
    step) are then out of the timed loop, as in a serving engine that plans step n + 1
    while the GPU runs step n."""

    def __init__(self, ts: TraceSpec, device="cuda", max_reqs: int | None = None):
        import torch

        from . import kvpaged as kp
        self.torch, self.kp = torch, kp
        self.ts, self.device = ts, device
        self.trace = make_trace(ts)
        self.pool = kp.KVPool(ts.pool_blocks, device=device)
        h = self.pool.handle
        n_shared = ts.shared_prefix // BLOCK_SIZE
        self.shared_blocks = [int(b) for b in kp.kv_block_alloc(h, n_shared)]
        longest = ts.shared_prefix + max(r.prompt_len for r in self.trace) + max(r.output_len for r in self.trace)
        self.width = -(-longest // BLOCK_SIZE) + 1
        self.max_reqs = max_reqs or ts.n_requests
        T = ts.budget
        self.q = torch.empty((T, 4096), dtype=torch.bfloat16, device=device)
        self.k_new = torch.empty((T, 1024), dtype=torch.bfloat16, device=device)
        self.v_new = torch.empty((T, 1024), dtype=torch.bfloat16, device=device)
        self.out = torch.empty((T, 4096), dtype=torch.bfloat16, device=device)
        self.ws = torch.empty(kp.paged_attention_workspace_size(h, self.max_reqs, T, longest), dtype=torch.uint8,
                              device=device)
        self._log = None   # block-manager calls of the current step, while recording
        self.sched = Scheduler(self.trace, ts, self.shared_blocks, self._alloc, self._ref, self._free)
        self._write_shared_prefix()
        self.step_ms = []
        self.step_tokens = []
        self.step_decode_bytes = []
        self.checks = []

    def _alloc(self, n):
        ids = self.kp.kv_block_alloc(self.pool.handle, n)
        if self._log is not None:
            self._log.append(("alloc", [int(b) for b in ids]))
        return ids

    def _ref(self, ids):
        self.kp.kv_block_ref(self.pool.handle, ids)
        if self._log is not None:
            self._log.append(("ref", [int(b) for b in ids]))

    def _free(self, ids):
        self.kp.kv_block_free(self.pool.handle, ids)
        if self._log is not None:
            self._log.append(("free", [int(b) for b in ids]))

    def _write_shared_prefix(self):
        torch, kp = self.torch, self.kp
        n = self.ts.shared_prefix
        if n == 0:
            return
        _, k, v = trace_rows(self.ts.seed, -1, 0, n)
        dev = self.device
        kk = torch.from_numpy(k.view(np.int16)).to(dev).view(torch.bfloat16)
        vv = torch.from_numpy(v.view(np.int16)).to(dev).view(torch.bfloat16)
        table = torch.tensor([self.shared_blocks], dtype=torch.int32, device=dev)
        kp.kv_append(self.pool.handle, kk, vv, torch.tensor([0, n], dtype=torch.int32, device=dev),
                     torch.zeros(1, dtype=torch.int32, device=dev), table)

    def _rows(self, plan: StepPlan):
        jobs = [(rs.req.rid, ctx, q) for rs, ctx, q in plan.entries]
        with ThreadPoolExecutor(16) as ex:
            parts = list(ex.map(lambda j: trace_rows(self.ts.seed, *j), jobs))
        return (np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]),
                np.concatenate([p[2] for p in parts]))

    def run(self, max_steps: int | None = None, check_every: int = 0, check_rows: int = 4, oracle=None,
            on_check=None, record: bool = False):
        """Replay the trace.  With check_every > 0, every check_every-th step a few rows are
        compared against `oracle` (a callable taking (q rows, K histories, V histories,
        cu, ctx) and returning fp64 outputs) through `on_check(step, got, want)`.  With
        record, every step is kept for `replay()`."""
        torch, kp = self.torch, self.kp
        dev = self.device
        stream = torch.cuda.current_stream(dev)
        evs = []
        h = self.pool.handle
        if record:
            self.recorded = []
        while not self.sched.finished() and (max_steps is None or self.sched.step < max_steps):
            pre = self._log = [] if record else None
            plan = self.sched.plan()
            if not plan.entries:
                post = self._log = [] if record else None
                self.sched.commit(plan)
                self._log = None
                if record:
                    self.recorded.append({"pre": pre, "post": post, "T": 0})
                continue
            R, T = len(plan.entries), plan.num_tokens
            if R > self.max_reqs:
                raise RuntimeError(f"step {plan.step}: {R} requests exceed the workspace sizing ({self.max_reqs})")
            cu = np.zeros(R + 1, np.int32)
            cu[1:] = np.cumsum([q for _, _, q in plan.entries])
            ctx = np.array([c for _, c, _ in plan.entries], np.int32)
            tables = np.stack([self.sched.table_row(rs, self.width) for rs, _, _ in plan.entries])
            q, k, v = self._rows(plan)
            self.q[:T].copy_(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16))
            self.k_new[:T].copy_(torch.from_numpy(k.view(np.int16)).view(torch.bfloat16))
            self.v_new[:T].copy_(torch.from_numpy(v.view(np.int16)).view(torch.bfloat16))
            cu_d = torch.from_numpy(cu).to(dev)
            ctx_d = torch.from_numpy(ctx).to(dev)
            tab_d = torch.from_numpy(tables).to(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            kp.kv_append(h, self.k_new[:T], self.v_new[:T], cu_d, ctx_d, tab_d)
            kp.paged_attention_step(h, self.q[:T], self.out[:T], cu_d, ctx_d, tab_d, int(max(cu[1:] - cu[:-1])),
                                    int(ctx.max()), 1.0 / math.sqrt(128.0), self.ws)
            e1.record(stream)
            evs.append((e0, e1))
            self.step_tokens.append(T)
            self.step_decode_bytes.append(sum(4096 * (c + 1) for (_, c, qq) in plan.entries if qq == 1))
            if record:
                self.recorded.append({"pre": pre, "T": T, "q": self.q[:T].clone(), "k": self.k_new[:T].clone(),
                                      "v": self.v_new[:T].clone(), "cu": cu_d, "ctx": ctx_d, "tab": tab_d,
                                      "max_q": int(max(cu[1:] - cu[:-1])), "max_ctx": int(ctx.max())})
            if check_every and oracle is not None and plan.step % check_every == 0:
                torch.cuda.synchronize(dev)
                got = self.out[:T].float().cpu().numpy().reshape(T, 32, 128)
                pick = np.unique(np.linspace(0, R - 1, min(R, check_rows)).round().astype(int))
                rows, ks, vs, cu_s, ctx_s = [], [], [], [0], []
                for i in pick:
                    rs, c, qq = plan.entries[i]
                    hk, hv = history(self.ts, rs)
                    hk = np.concatenate([hk, k[cu[i]:cu[i + 1]]])
                    hv = np.concatenate([hv, v[cu[i]:cu[i + 1]]])
                    ks.append(hk)
                    vs.append(hv)
                    rows.append(q[cu[i]:cu[i + 1]])
                    cu_s.append(cu_s[-1] + qq)
                    ctx_s.append(c)
                want = oracle(np.concatenate(rows), ks, vs, np.array(cu_s, np.int32), np.array(ctx_s, np.int32))
                sel = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in pick])
                on_check(plan.step, got[sel], want)
                self.checks.append(plan.step)
            post = self._log = [] if record else None
            self.sched.commit(plan)
            self._log = None
            if record:
                self.recorded[-1]["post"] = post
        torch.cuda.synchronize(dev)
        self.step_ms = [a.elapsed_time(b) for a, b in evs]
        return self

    def replay(self, timing_launches: int = 0) -> dict:
        """Serve the recorded steps again on a fresh pool, back to back: per step the
        block-manager calls made before it (runs of one kind merged into one call: the
        allocator hands out and takes back ids in call order), kv_append and
        paged_attention_step on the recorded device inputs, then the calls made after it.
        Returns the tokens and the GPU time of the whole replay (one pair of events around
        it, so host time between steps counts when the GPU waits for it).  With
        timing_launches > 0 the library also times each of its kernel launches (events
        around each, which stops their overlap) and the result holds the per-kernel sums."""
        torch, kp = self.torch, self.kp
        dev = self.device
        stream = torch.cuda.current_stream(dev)
        shared = list(self.shared_blocks)
        self.pool.close()
        self.pool = kp.KVPool(self.ts.pool_blocks, device=dev)
        h = self.pool.handle
        got = [int(b) for b in kp.kv_block_alloc(h, len(shared))]
        if got != shared:
            raise RuntimeError("replay: the fresh pool handed out other shared-prefix blocks")
        self._write_shared_prefix()
        if timing_launches:
            kp.kv_pool_enable_timing(h, timing_launches)

        def apply(ops):
            i = 0
            while i < len(ops):
                kind, ids = ops[i][0], list(ops[i][1])
                j = i + 1
                while j < len(ops) and ops[j][0] == kind:
                    ids += ops[j][1]
                    j += 1
                if kind == "alloc":
                    if [int(b) for b in kp.kv_block_alloc(h, len(ids))] != ids:
                        raise RuntimeError("replay: the allocator handed out other blocks than recorded")
                elif kind == "ref":
                    kp.kv_block_ref(h, ids)
                else:
                    kp.kv_block_free(h, ids)
                i = j

        scale = 1.0 / math.sqrt(128.0)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tokens = 0
        e0.record(stream)
        for rec in self.recorded:
            apply(rec["pre"])
            T = rec["T"]
            if T:
                kp.kv_append(h, rec["k"], rec["v"], rec["cu"], rec["ctx"], rec["tab"])
                kp.paged_attention_step(h, rec["q"], self.out[:T], rec["cu"], rec["ctx"], rec["tab"], rec["max_q"],
                                        rec["max_ctx"], scale, self.ws)
                tokens += T
            apply(rec["post"])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1)
        res = {"steps": sum(1 for r in self.recorded if r["T"]), "tokens": tokens, "gpu_ms": ms,
               "tokens_per_s": tokens / (ms / 1e3) if ms > 0 else 0.0}
        if timing_launches:
            res["kernels"] = kp.kv_pool_read_timing(h)
            kp.kv_pool_enable_timing(h, 0)
        st = kp.kv_pool_get_error(h)
        if st != (0, 0):
            raise RuntimeError(f"replay: device error word {st}")
        return res

    def summary(self) -> dict:
        ms = np.array(self.step_ms)
        tok = int(np.sum(self.step_tokens))
        return {"steps": len(ms), "tokens": tok, "gpu_ms": float(ms.sum()),
                "tokens_per_s": tok / (ms.sum() / 1e3) if len(ms) else 0.0,
                "step_ms_p50": float(np.percentile(ms, 50)) if len(ms) else None,
                "step_ms_p90": float(np.percentile(ms, 90)) if len(ms) else None,
                "step_ms_p99": float(np.percentile(ms, 99)) if len(ms) else None,
                "decode_bytes": int(np.sum(self.step_decode_bytes)),
                "requests_done": len(self.sched.done)}

    def close(self):
        self.pool.close()
