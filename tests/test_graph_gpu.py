"""A fixed-shape step captured in a CUDA graph and replayed (launch overhead cut for
repeated steps of the same shape; page "Continuous Batching 深入实现", section "一次完整
decode step 的 timeline", names the graph launch) computes what the method defines: every
replay's output matches the fp64 oracle at the parity tolerance, and the pool after the
replays is the oracle's cache write bit for bit (re-appending the same rows into the same
slots changes nothing)."""
import numpy as np
import pytest

import oracle
from continuous_batching_paged_step_gb300 import workloads as wl

import parity_helpers as ph

pytestmark = pytest.mark.gpu

NAN_BITS = 0x7FC1


def test_graph_replay_matches_oracle():
    import torch
    from continuous_batching_paged_step_gb300 import build
    build.build()
    from continuous_batching_paged_step_gb300 import runner
    inp = wl.make_inputs(wl.small_mixed_step())
    want = oracle.step_reference(inp)
    step = runner.PagedStep(inp, pool_fill_bits=NAN_BITS, poison_workspace=True)
    try:
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            step.run(stream=stream)                 # device state made, nothing pending
        stream.synchronize()
        direct = step.out.clone()
        g = torch.cuda.CUDAGraph()
        step.out.fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            step.run(stream=stream)
        for _ in range(3):
            step.out.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            got = step.out_f32()
            assert np.isfinite(got).all(), "replay left rows unwritten"
            mx, mn = ph.errors(got, want)
            assert mx <= ph.MAX_ABS and mn <= ph.MEAN_ABS, f"replay vs oracle: max {mx:.3e} mean {mn:.3e}"
            assert torch.equal(step.out, direct)     # and the same bits as a direct call
        assert step.error() == (0, 0)
        k, v = ph.pool_bits(step)
        ok_k, ok_v = ph.oracle_pool(inp, NAN_BITS)
        assert np.array_equal(k, ok_k) and np.array_equal(v, ok_v), "pool differs from the oracle's cache write"
    finally:
        step.close()
