"""GPU test of paged_attention_step_noalloc.

The allocation-free variant of the attention step serves callers that cannot allocate
device memory at step time (an engine that has handed all free device memory to its KV
pool, or a serving loop that must not call cudaMalloc/cudaFree because they can
synchronise the device): its scratch lives in a fixed array inside the library instead
of a caller workspace.  Through the C ABI, two calls in a row must give what the
workspace-based paged_attention_step gives on the same step, within the tolerance of the
parity tests.  This file is collected last on purpose: it shares nothing with the other
tests and passes alone or after them.
"""
import ctypes

import numpy as np
import pytest

from continuous_batching_paged_step_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3


@pytest.fixture(scope="module")
def mods():
    from continuous_batching_paged_step_gb300 import build
    build.build()
    from continuous_batching_paged_step_gb300 import kvpaged, runner
    return kvpaged, runner


def test_noalloc_step_matches_workspace_step_twice(mods):
    import torch
    kp, runner = mods
    inp = wl.make_inputs(wl.small_mixed_step())        # prefill chunks and decode rows
    step = runner.PagedStep(inp)                        # its kv_append makes the pool's device state
    try:
        step.run()                                      # workspace-based step
        want = step.out.float().cpu().numpy()
        assert step.error() == (0, 0)
        before = torch.cuda.memory_allocated()
        for _ in range(2):
            out = torch.full_like(step.q, float("nan"))
            kp.paged_attention_step_noalloc(step.pool.handle, step.q, out, step.cu_seqlens_q, step.context_lens,
                                            step.block_tables, step.max_q_len, step.max_context_len,
                                            step.softmax_scale)
            torch.cuda.synchronize()
            got = out.float().cpu().numpy()
            assert np.isfinite(got).all()
            err = np.abs(got.astype(np.float64) - want)
            assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (err.max(), err.mean())
            del out
        assert step.error() == (0, 0)
        assert torch.cuda.memory_allocated() == before
    finally:
        step.close()


def test_noalloc_rejects_oversize_and_pool_without_device_state(mods):
    import torch
    kp, _ = mods
    lib = kp.lib
    assert kp.paged_attention_noalloc_capacity() == 32 << 20
    fake = ctypes.c_void_p(0x10000)
    # a fresh pool has no device state yet: the allocation-free call refuses to make it
    pool = kp.KVPool(8)
    try:
        st = lib.paged_attention_step_noalloc(pool.handle, fake, fake, fake, fake, fake, 1, 1, 1, 32, 1, 0,
                                              0.088, None)
        assert st == -1
        # scratch for a million requests cannot fit in the fixed array: rejected up front
        st = lib.paged_attention_step_noalloc(pool.handle, fake, fake, fake, fake, fake, 1, 1_000_000, 1_000_000,
                                              32, 1, 0, 0.088, None)
        assert st == -8
    finally:
        pool.close()
    torch.cuda.synchronize()
