"""Device-detected errors: the kernels set bits in the pool's error word, skip the
offending write or request, and still produce every other output.  No test faults,
traps or hangs the GPU: every bad input here is one the kernels check for."""
import numpy as np
import pytest

import oracle
from continuous_batching_paged_step_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    from continuous_batching_paged_step_gb300 import build
    build.build()
    from continuous_batching_paged_step_gb300 import kvpaged, runner
    return kvpaged, runner


def _small():
    return wl.StepSpec("err", q_lens=[1, 1, 20], ctx_lens=[40, 17, 16], num_blocks=32, seed=31)


def test_write_into_shared_block_is_refused(mods):
    kp, runner = mods
    inp = wl.make_inputs(_small())
    step = runner.PagedStep(inp)
    try:
        # request 0 (40 cached + 1 new) writes position 40 into its third block; share it
        b = int(inp.block_tables[0, 40 // 16])
        kp.kv_block_ref(step.pool.handle, [b])
        before = step.pool.k_cache[b].clone()
        step.append()
        st, bits = step.error()
        assert st == -4
        assert bits & kp.ERRBIT_SHARED_WRITE
        assert step.pool.k_cache[b].equal(before)         # the write was skipped
        # once the share is dropped the same append goes through
        kp.kv_block_free(step.pool.handle, [b])
        step.append()
        assert step.error() == (0, 0)
    finally:
        step.close()


@pytest.mark.parametrize("mixed", [False, True], ids=["two_kernels", "mixed_kernel"])
@pytest.mark.parametrize("bad", [1, 2], ids=["decode_row", "prefill_chunk"])
def test_bad_block_id_is_flagged_and_others_survive(mods, bad, mixed):
    kp, runner = mods
    import torch
    inp = wl.make_inputs(_small())
    step = runner.PagedStep(inp, mixed=mixed)
    try:
        step.run()
        good = step.out_f32()
        assert step.error() == (0, 0)
        # corrupt one entry of request `bad`'s table (a cached page it reads, not one it
        # writes): request 1 is a decode row, request 2 a prefill chunk
        step.block_tables[bad, 0] = 10 ** 6
        step.out.zero_()
        step.attend()
        st, bits = step.error()
        assert bits & kp.ERRBIT_BAD_BLOCK
        got = step.out_f32()
        cu = inp.cu_seqlens_q
        for r in (0, 1, 2):
            if r == bad:
                continue
            s, e = cu[r], cu[r + 1]
            assert np.array_equal(got[s:e], good[s:e])
        step.block_tables[bad, 0] = int(inp.block_tables[bad, 0])
    finally:
        step.close()


def test_inconsistent_metadata_is_flagged(mods):
    kp, runner = mods
    import torch
    inp = wl.make_inputs(_small())
    step = runner.PagedStep(inp)
    try:
        # cu_seqlens_q that does not end at num_tokens: no work at all, BAD_META
        bad_cu = step.cu_seqlens_q.clone()
        bad_cu[-1] += 1
        kp.paged_attention_step(step.pool.handle, step.q, step.out, bad_cu, step.context_lens, step.block_tables,
                                step.max_q_len, step.max_context_len, step.softmax_scale, step.workspace)
        assert step.error()[1] & kp.ERRBIT_BAD_META
        # a context length above the declared maximum: that request is skipped
        kp.paged_attention_step(step.pool.handle, step.q, step.out, step.cu_seqlens_q, step.context_lens,
                                step.block_tables, step.max_q_len, 20, step.softmax_scale, step.workspace)
        assert step.error()[1] & kp.ERRBIT_BAD_META
        # a row whose position falls past the table width: kv_append flags and skips it
        narrow = step.block_tables[:, :2].contiguous()
        kp.kv_append(step.pool.handle, step.k_new, step.v_new, step.cu_seqlens_q, step.context_lens, narrow)
        assert step.error()[1] & kp.ERRBIT_BAD_META
    finally:
        step.close()


def test_host_argument_errors(mods):
    kp, runner = mods
    import torch
    inp = wl.make_inputs(_small())
    step = runner.PagedStep(inp)
    try:
        tiny_ws = torch.empty(256, dtype=torch.uint8, device="cuda")
        with pytest.raises(kp.KVPError) as e:
            kp.paged_attention_step(step.pool.handle, step.q, step.out, step.cu_seqlens_q, step.context_lens,
                                    step.block_tables, step.max_q_len, step.max_context_len, step.softmax_scale,
                                    tiny_ws)
        assert e.value.status == -8
        with pytest.raises(kp.KVPError) as e:
            kp.paged_attention_step(step.pool.handle, step.q, step.out, step.cu_seqlens_q, step.context_lens,
                                    step.block_tables, step.max_q_len, step.max_context_len, -1.0, step.workspace)
        assert e.value.status == -1
        assert step.error() == (0, 0)      # nothing was launched
    finally:
        step.close()


def test_bounded_wait_gives_up_and_the_context_survives(mods):
    # A wait that nothing completes gives up after its limit and reports it; the GPU
    # context stays usable (a full step afterwards is still correct).
    import time
    kp, runner = mods
    t0 = time.perf_counter()
    assert kp.kvp_selftest_bounded_wait(50_000_000) == -9          # KVP_E_TIMEOUT after ~50 ms
    assert time.perf_counter() - t0 < 5.0
    inp = wl.make_inputs(wl.tiny_p5_step())
    step = runner.PagedStep(inp)
    try:
        step.run()
        assert step.error() == (0, 0)
        want = oracle.step_reference(inp)
        assert np.abs(step.out_f32() - want).max() <= 2e-2
    finally:
        step.close()
