"""A short trace replayed on the GPU: every step is kv_append + paged_attention_step on a
pool whose shared system-prompt blocks are referenced by every request.  Sampled rows of
sampled steps are compared with the oracle, which rebuilds each request's history from
the seeded chunks (never from the pool)."""
import numpy as np
import pytest

import oracle
from continuous_batching_paged_step_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3


def test_short_trace_against_oracle():
    from continuous_batching_paged_step_gb300 import build
    build.build()
    from continuous_batching_paged_step_gb300 import kvpaged as kp
    from continuous_batching_paged_step_gb300.trace import TraceRunner
    ts = wl.TraceSpec(name="short", n_requests=40, arrivals_per_step=3.0, shared_prefix=64, prompt_median=60,
                      prompt_cap=400, output_median=12, output_range=(10, 40), budget=256, pool_blocks=4096, seed=21)
    tr = TraceRunner(ts)
    errs = []

    def on_check(step, got, want):
        assert np.isfinite(got).all(), f"step {step}: non-finite output"
        e = np.abs(got.astype(np.float64) - want)
        assert e.max() <= MAX_ABS and e.mean() <= MEAN_ABS, (step, e.max(), e.mean())
        errs.append(e.max())

    def ref(q, ks, vs, cu, ctx):
        return oracle.attention_reference(q, ks, vs, cu, ctx, 32, 8, 128)

    try:
        free0 = kp.kv_pool_num_free(tr.pool.handle)
        tr.run(check_every=4, check_rows=5, oracle=ref, on_check=on_check)
        s = tr.summary()
        assert s["requests_done"] == ts.n_requests
        assert len(tr.checks) >= 5
        assert kp.kv_pool_get_error(tr.pool.handle) == (0, 0)
        # every request returned its blocks; the shared prefix is held once
        assert kp.kv_pool_num_free(tr.pool.handle) == free0
        assert all(kp.kv_block_refcount(tr.pool.handle, b) == 1 for b in tr.shared_blocks)
    finally:
        tr.close()


def test_replay_matches_the_served_run():
    # The recorded steps served again on a fresh pool (the benchmark's timed replay) give
    # bit-identical outputs, hand out the same blocks and leave the pool as the served run did.
    from continuous_batching_paged_step_gb300 import build
    build.build()
    import torch
    from continuous_batching_paged_step_gb300 import kvpaged as kp
    from continuous_batching_paged_step_gb300.trace import TraceRunner
    ts = wl.TraceSpec(name="short-replay", n_requests=30, arrivals_per_step=3.0, shared_prefix=32, prompt_median=50,
                      prompt_cap=300, output_median=12, output_range=(10, 30), budget=192, pool_blocks=2048, seed=33)
    tr = TraceRunner(ts)
    try:
        tr.run(max_steps=25, record=True)
        last = max(i for i, r in enumerate(tr.recorded) if r["T"])
        T = tr.recorded[last]["T"]
        served_out = tr.out[:T].clone()
        free_served = kp.kv_pool_num_free(tr.pool.handle)
        res = tr.replay()
        torch.cuda.synchronize()
        assert res["steps"] == sum(1 for r in tr.recorded if r["T"])
        assert res["tokens"] == sum(r["T"] for r in tr.recorded)
        assert torch.equal(tr.out[:T].view(torch.int16), served_out.view(torch.int16))
        assert kp.kv_pool_num_free(tr.pool.handle) == free_served
    finally:
        tr.close()
