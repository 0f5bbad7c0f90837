"""A fixed-shape step captured in a CUDA graph and replayed (launch overhead cut for
repeated steps of the same shape) gives what direct calls give."""
import numpy as np
import pytest

from continuous_batching_paged_step_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_graph_replay_matches_direct_calls():
    import torch
    from continuous_batching_paged_step_gb300 import build
    build.build()
    from continuous_batching_paged_step_gb300 import runner
    inp = wl.make_inputs(wl.small_mixed_step())
    step = runner.PagedStep(inp)
    try:
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            step.run(stream=stream)                 # device state made, nothing pending
        stream.synchronize()
        want = step.out.clone()
        g = torch.cuda.CUDAGraph()
        step.out.zero_()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            step.run(stream=stream)
        for _ in range(3):
            step.out.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(step.out, want)
        assert step.error() == (0, 0)
    finally:
        step.close()
