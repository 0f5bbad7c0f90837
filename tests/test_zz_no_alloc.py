"""GPU test of paged_attention_step_noalloc.

The allocation-free variant of the attention step serves callers that cannot allocate
device memory at step time (an engine that has handed all free device memory to its KV
pool, or a serving loop that must not call cudaMalloc/cudaFree because they can
synchronise the device): its scratch lives in a fixed array inside the library instead
of a caller workspace.  Through the C ABI, calls in a row must match the fp64 oracle at
the parity tolerance and the workspace-based paged_attention_step on the same step, and
the device's free memory must not change across them.  This file is collected last on
purpose: it shares nothing with the other tests and passes alone or after them.
"""
import ctypes

import numpy as np
import pytest

import oracle
from continuous_batching_paged_step_gb300 import workloads as wl

import parity_helpers as ph

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    from continuous_batching_paged_step_gb300 import build
    build.build()
    from continuous_batching_paged_step_gb300 import kvpaged, runner
    return kvpaged, runner


def test_noalloc_step_matches_oracle_and_workspace_step(mods):
    import torch
    kp, runner = mods
    inp = wl.make_inputs(wl.small_mixed_step())        # prefill chunks and decode rows
    want = oracle.step_reference(inp)
    step = runner.PagedStep(inp)                        # its kv_append makes the pool's device state
    try:
        step.run()                                      # workspace-based step
        ws_out = step.out.float().cpu().numpy().reshape(want.shape)
        assert step.error() == (0, 0)
        outs = [torch.full_like(step.q, float("nan")) for _ in range(3)]

        def call(out):
            kp.paged_attention_step_noalloc(step.pool.handle, step.q, out, step.cu_seqlens_q, step.context_lens,
                                            step.block_tables, step.max_q_len, step.max_context_len,
                                            step.softmax_scale)

        # The first call looks the scratch array's address up; with CUDA's lazy module
        # loading that is also when the array is placed on the device.
        call(outs[0])
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        alloc0 = torch.cuda.memory_allocated()
        call(outs[1])
        call(outs[2])                                   # two calls in a row
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        assert free1 == free0, f"device free memory changed by {free0 - free1} bytes across the calls"
        assert torch.cuda.memory_allocated() == alloc0
        for i, out in enumerate(outs):
            got = out.float().cpu().numpy().reshape(want.shape)
            assert np.isfinite(got).all(), f"call {i}: rows left unwritten"
            mx, mn = ph.errors(got, want)
            assert mx <= ph.MAX_ABS and mn <= ph.MEAN_ABS, f"call {i} vs oracle: max {mx:.3e} mean {mn:.3e}"
            mx, mn = ph.errors(got, ws_out)
            assert mx <= ph.MAX_ABS and mn <= ph.MEAN_ABS, f"call {i} vs workspace step: max {mx:.3e} mean {mn:.3e}"
        assert step.error() == (0, 0)
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


def test_noalloc_request_limit(mods):
    # The fixed array holds the scratch of a decode step of about 990 requests: each
    # request and each of the decode kernel's up to 1,024 pieces has a slot of split-KV
    # partials (32 heads x 128 fp32 plus 32 (max, sum) pairs).  Host arithmetic only.
    kp, _ = mods
    lib = kp.lib
    h = ctypes.c_void_p()
    # a pool handle over two dummy (aligned, never touched) addresses: the size query is host arithmetic
    assert lib.kv_pool_create(8, 16, 8, 128, 1, ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000),
                              ctypes.byref(h)) == 0
    try:
        cap = kp.paged_attention_noalloc_capacity()
        fits = [n for n in (900, 980, 990, 991, 992, 1000, 1100)
                if lib.paged_attention_workspace_size(h, n, n, 32, 8192) <= cap]
        assert fits == [900, 980, 990, 991]
    finally:
        lib.kv_pool_destroy(h)
