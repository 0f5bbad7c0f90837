"""Whole-block operations of the block manager on the GPU: copy-on-write of a shared
block (page "11.2 连续批处理与 PagedAttention", section 11.2.3, sharing within one
request) and swapping a request's blocks out to host memory and back (page "Continuous
Batching 深入实现", section "第四层").  Copies are checked bit for bit; the flows end in
an attention step checked against the oracle."""
import numpy as np
import pytest

import oracle
from continuous_batching_paged_step_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

BLOCK_U16 = 8 * 16 * 128     # bf16 values in one block of K (or V)


@pytest.fixture(scope="module")
def mods():
    from continuous_batching_paged_step_gb300 import build
    build.build()
    from continuous_batching_paged_step_gb300 import kvpaged, runner
    return kvpaged, runner


def _random_pool(kp, num_blocks, seed):
    import torch
    pool = kp.KVPool(num_blocks)
    g = torch.Generator(device="cuda").manual_seed(seed)
    for t in (pool.k_cache, pool.v_cache):
        t.view(torch.int16).copy_(torch.randint(-32768, 32767, t.shape, generator=g, device="cuda",
                                                dtype=torch.int32).to(torch.int16))
    return pool


def _bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy()


def test_cow_copies_only_shared_blocks(mods):
    kp, _ = mods
    import torch
    pool = _random_pool(kp, 64, 1)
    h = pool.handle
    try:
        x, y, z = (int(b) for b in kp.kv_block_alloc(h, 3))
        kp.kv_block_ref(h, [x])            # refcount 2
        kp.kv_block_ref(h, [z, z])         # refcount 3
        k0, v0 = _bits(pool.k_cache), _bits(pool.v_cache)
        out = [int(b) for b in kp.kv_block_cow(h, [x, y, z, z])]
        torch.cuda.synchronize()
        assert out[1] == y                                   # not shared: no copy
        assert len({out[0], out[2], out[3], x, y, z}) == 6   # three fresh blocks
        assert [kp.kv_block_refcount(h, b) for b in (x, y, z)] == [1, 1, 1]
        assert all(kp.kv_block_refcount(h, b) == 1 for b in (out[0], out[2], out[3]))
        k1, v1 = _bits(pool.k_cache), _bits(pool.v_cache)
        for src, dst in ((x, out[0]), (z, out[2]), (z, out[3])):
            assert np.array_equal(k1[dst], k0[src]) and np.array_equal(v1[dst], v0[src])
        untouched = [b for b in range(64) if b not in (out[0], out[2], out[3])]
        assert np.array_equal(k1[untouched], k0[untouched]) and np.array_equal(v1[untouched], v0[untouched])
        assert kp.kv_pool_get_error(h) == (0, 0)
    finally:
        pool.close()


def _bf16(rng, shape):
    return wl.f32_to_bf16_bits(rng.standard_normal(int(np.prod(shape)), dtype=np.float32)).reshape(shape)


def test_cow_then_append_parallel_sampling(mods):
    """Two output sequences of one request share a 20-token prompt (block 0 full, block 1
    holding 4 tokens).  Sequence A copies block 1 before writing token 20 into it; B then
    writes its own token 20 into the original.  Each decode row must see the prompt plus
    its own token only."""
    kp, _ = mods
    import torch
    rng = np.random.default_rng(7)
    n_prompt = 20
    kpr, vpr = _bf16(rng, (n_prompt, 1024)), _bf16(rng, (n_prompt, 1024))
    q, kn, vn = _bf16(rng, (2, 4096)), _bf16(rng, (2, 1024)), _bf16(rng, (2, 1024))
    pool = kp.KVPool(32)
    h = pool.handle
    dev = "cuda"

    def t16(a):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

    def t32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    try:
        b0, b1 = (int(b) for b in kp.kv_block_alloc(h, 2))
        kp.kv_append(h, t16(kpr), t16(vpr), t32([0, n_prompt]), t32([0]), t32([[b0, b1]]))
        kp.kv_block_ref(h, [b0, b1])                      # both sequences hold the prompt
        b1a = int(kp.kv_block_cow(h, [b1])[0])            # A writes into block 1: copy it first
        assert b1a != b1 and kp.kv_block_refcount(h, b1) == 1 and kp.kv_block_refcount(h, b0) == 2
        tables = t32([[b0, b1a], [b0, b1]])
        cu, ctx = t32([0, 1, 2]), t32([n_prompt, n_prompt])
        kp.kv_append(h, t16(kn), t16(vn), cu, ctx, tables)
        out = torch.zeros(2, 4096, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(kp.paged_attention_workspace_size(h, 2, 2, n_prompt), dtype=torch.uint8, device=dev)
        kp.paged_attention_step(h, t16(q), out, cu, ctx, tables, 1, n_prompt, 1 / np.sqrt(128), ws)
        assert kp.kv_pool_get_error(h) == (0, 0)
        spec = wl.StepSpec("cow", q_lens=[1, 1], ctx_lens=[n_prompt, n_prompt], num_blocks=32, seed=0)
        inp = wl.StepInputs(spec=spec, q=q, k_new=kn, v_new=vn, k_prior=[kpr, kpr], v_prior=[vpr, vpr],
                            cu_seqlens_q=np.array([0, 1, 2], np.int32),
                            context_lens=np.array([n_prompt, n_prompt], np.int32),
                            block_tables=np.array([[b0, b1a], [b0, b1]], np.int32),
                            block_order=np.array([b0, b1, b1a], np.int32))
        want = oracle.step_reference(inp)
        got = out.float().cpu().numpy().reshape(2, 32, 128)
        err = np.abs(got - want)
        assert err.max() <= 2e-2 and err.mean() <= 2e-3
        # the copy kept the prompt's 4 tokens of block 1; slot 4 differs between A and B
        kb = pool.k_cache.view(torch.int16).cpu().numpy()
        assert np.array_equal(kb[b1a][:, :4], kb[b1][:, :4])
        assert np.array_equal(kb[b1a][:, 4].reshape(-1), kn[0].view(np.int16))
        assert np.array_equal(kb[b1][:, 4].reshape(-1), kn[1].view(np.int16))
    finally:
        pool.close()


def test_swap_roundtrip_many_blocks(mods):
    """More blocks than one launch carries (1024): out to host and back, bit for bit."""
    kp, _ = mods
    import torch
    nb = 3200
    pool = _random_pool(kp, nb, 3)
    h = pool.handle
    try:
        ids = kp.kv_block_alloc(h, 1500)
        rng = np.random.default_rng(5)
        ids = ids[rng.permutation(ids.size)]
        k0, v0 = _bits(pool.k_cache), _bits(pool.v_cache)
        hk = torch.empty(ids.size * kp.BLOCK_BYTES, dtype=torch.uint8).pin_memory()
        hv = torch.empty_like(hk).pin_memory()
        kp.kv_blocks_swap_out(h, ids, hk, hv)
        torch.cuda.synchronize()
        assert kp.kv_pool_num_free(h) == nb
        hk16, hv16 = hk.view(torch.int16).numpy().reshape(ids.size, -1), hv.view(torch.int16).numpy().reshape(ids.size, -1)
        assert np.array_equal(hk16, k0[ids].reshape(ids.size, -1))
        assert np.array_equal(hv16, v0[ids].reshape(ids.size, -1))
        # hand the freed blocks out again and overwrite them, then swap back in elsewhere
        held = kp.kv_block_alloc(h, 1500)
        pool.k_cache[torch.from_numpy(held.astype(np.int64)).cuda()] = 0
        new = kp.kv_blocks_swap_in(h, hk, hv, ids.size)
        torch.cuda.synchronize()
        assert not set(new.tolist()) & set(held.tolist())
        k1, v1 = _bits(pool.k_cache), _bits(pool.v_cache)
        assert np.array_equal(k1[new].reshape(ids.size, -1), hk16)
        assert np.array_equal(v1[new].reshape(ids.size, -1), hv16)
        assert all(kp.kv_block_refcount(h, int(b)) == 1 for b in new)
    finally:
        pool.close()


def test_preempt_by_swap_then_resume(mods):
    """A decode request is preempted (its blocks swapped out and reused by others), then
    resumed into different blocks: the resumed step equals the oracle."""
    kp, runner = mods
    import torch
    spec = wl.StepSpec("swap", q_lens=[1, 1, 9], ctx_lens=[100, 33, 20], num_blocks=96, seed=11)
    inp = wl.make_inputs(spec)
    step = runner.PagedStep(inp)
    h = step.pool.handle
    try:
        n0 = spec.blocks_needed(0)
        mine = inp.block_tables[0, :n0].copy()
        hk = torch.empty(n0 * kp.BLOCK_BYTES, dtype=torch.uint8).pin_memory()
        hv = torch.empty_like(hk).pin_memory()
        kp.kv_blocks_swap_out(h, mine, hk, hv)
        # another request takes the freed blocks and writes over them
        other = kp.kv_block_alloc(h, n0)
        assert sorted(other.tolist()) == sorted(mine.tolist())
        step.pool.k_cache[torch.from_numpy(other.astype(np.int64)).cuda()] = 1.0
        step.pool.v_cache[torch.from_numpy(other.astype(np.int64)).cuda()] = -1.0
        back = kp.kv_blocks_swap_in(h, hk, hv, n0)
        assert not set(back.tolist()) & set(other.tolist())
        step.block_tables[0, :n0] = torch.from_numpy(back.astype(np.int32)).cuda()
        step.run()
        assert step.error() == (0, 0)
        got = step.out_f32()
        want = oracle.step_reference(inp)
        err = np.abs(got - want)
        assert err.max() <= 2e-2 and err.mean() <= 2e-3
    finally:
        step.close()
