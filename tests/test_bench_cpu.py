"""The benchmark's host side, on CPU: the reference arm's JSON line (the CPU oracle timed
on a sample of a workload) and the row sampling both oracle timings use."""
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    r = _bench("--impl", "reference", "--config", "tiny", "--steps", "4", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["dtype"] == "f64" and d["data"] == "synthetic"
    assert d["steps"] == 4 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny-3req"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_stay_silent():
    r = _bench("--impl", "reference", "--config", "tiny", "--steps", "4", "--warmup", "3",
               env_extra={"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_oracle_rows_are_spread_over_the_step():
    import bench
    from continuous_batching_paged_step_gb300 import workloads as wl
    spec = wl.mixed_step()
    T = spec.num_tokens
    decode_rows = sum(1 for q in spec.q_lens if q == 1)
    for n in (1, 16, 64, 300, T, 5 * T):
        rows = bench.oracle_sample_rows(T, n)
        assert len(rows) == min(n, T)
        assert np.all(np.diff(rows) > 0) and rows[0] >= 0 and rows[-1] < T
    # decode rows (packed first here) enter in proportion to their share of the step
    rows = bench.oracle_sample_rows(T, 272)
    share = np.count_nonzero(rows < decode_rows) / len(rows)
    assert abs(share - decode_rows / T) < 0.02
    # successive samples start at different offsets and together cover every row
    seen = set()
    for shift in range(64):
        seen.update(int(x) for x in bench.oracle_sample_rows(T, 34, shift))
    assert len(seen) == T


def test_oracle_timing_repeats_until_the_requested_time():
    import bench
    n, wall, passes = bench.time_oracle("tiny", 4, min_seconds=0.05)
    assert passes >= 1 and wall >= 0.05 and n == 4 * passes
    n1, _, p1 = bench.time_oracle("tiny", 100)   # more rows than the step has: the whole step, once
    assert p1 == 1 and n1 == 7


def test_oracle_tasks_cover_the_sample_once():
    import bench
    from continuous_batching_paged_step_gb300 import workloads as wl
    spec = wl.chunked_prefill_step()
    cu = np.concatenate([[0], np.cumsum(spec.q_lens)])
    rows = bench.oracle_sample_rows(spec.num_tokens, 3000)
    tasks = bench.oracle_tasks(cu, spec.ctx_lens, rows, 16)
    flat = sorted(x for t in tasks for x in t)
    assert flat == sorted(int(x) for x in rows)
    for t in tasks:   # each task holds rows of one request
        reqs = set(int(r) for r in np.searchsorted(cu, t, side="right") - 1)
        assert len(reqs) == 1
    cost = [sum(spec.ctx_lens[int(np.searchsorted(cu, x, side="right") - 1)] + x - cu[int(np.searchsorted(cu, x, side="right") - 1)] + 1
                for x in t) for t in tasks]
    assert cost == sorted(cost, reverse=True)          # handed out longest first


def test_oracle_pool_matches_one_process():
    import bench
    rows = bench.oracle_sample_rows(7, 7)
    t = bench.OracleTimer("tiny", workers=2)
    try:
        n, w = t.time_rows(rows)
    finally:
        t.close()
    assert n == 7 and w > 0 and t.workers == 2
