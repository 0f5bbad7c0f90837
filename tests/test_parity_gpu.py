"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

kv_append and block-table indexing must be bit-exact; attention outputs (bf16) must be
within max-abs 2e-2 and mean-abs 2e-3 of the oracle.  Pools are pre-filled with a NaN
bit pattern, so a kernel that reads a slot it must not read shows up as NaN.
"""
import numpy as np
import pytest

import oracle
from continuous_batching_paged_step_gb300 import workloads as wl

import parity_helpers as ph

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3
NAN_BITS = 0x7FC1          # a bf16 quiet NaN used to fill pools before a test


@pytest.fixture(scope="module")
def runner():
    from continuous_batching_paged_step_gb300 import build
    build.build()
    from continuous_batching_paged_step_gb300 import runner as r
    return r


def _compare(got, want, rows=None, what=""):
    if rows is not None:
        got, want = got[rows], want[rows]
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got.astype(np.float64) - want)
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= MAX_ABS, f"{what}: max-abs {err.max():.3e} at {worst}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean-abs {err.mean():.3e}"
    return err.max(), err.mean()


def _run_full_check(runner, spec, ctas=None, mixed=False):
    # mixed: the mixed step kernel (one grid for decode rows and prefill tiles)
    inp = wl.make_inputs(spec)
    step = runner.PagedStep(inp, pool_fill_bits=NAN_BITS, decode_ctas=ctas, poison_workspace=True, mixed=mixed)
    try:
        step.run()
        st, bits = step.error()
        assert (st, bits) == (0, 0)
        k, v = ph.pool_bits(step)
        ok_k, ok_v = ph.oracle_pool(inp, NAN_BITS)
        assert np.array_equal(k, ok_k) and np.array_equal(v, ok_v), "pool differs from the oracle's cache write"
        return _compare(step.out_f32(), oracle.step_reference(inp), what=spec.name)
    finally:
        step.close()


@pytest.mark.parametrize("mixed", [False, True], ids=["two_kernels", "mixed_kernel"])
def test_three_request_example(runner, mixed):
    # page "11.2 连续批处理与 PagedAttention", section 11.2.2: R1 prefill 5 (nothing cached),
    # R2 decode with 7 cached, R3 decode with 3 cached; 64-block pool
    _run_full_check(runner, wl.tiny_p5_step(), mixed=mixed)


@pytest.mark.parametrize("mixed", [False, True], ids=["two_kernels", "mixed_kernel"])
def test_small_mixed_step_all_rows(runner, mixed):
    # prefill chunks spanning several 32-token q tiles with ragged tails, one of them after
    # a cached prefix that ends mid-block; decode rows with varied contexts
    _run_full_check(runner, wl.small_mixed_step(), mixed=mixed)


@pytest.mark.parametrize("ctas", [1, 7, 0, 1024])
def test_decode_split_and_combine(runner, ctas):
    # one CTA (no split), a few CTAs (most rows split across two), one per SM, and more
    # CTAs than blocks (every row split block by block; idle CTAs)
    spec = wl.small_mixed_step(seed=77, n_decode=20, chunks=(), ctx_range=(0, 1500), num_blocks=4096)
    _run_full_check(runner, spec, ctas=ctas)


@pytest.mark.parametrize("mixed", [False, True], ids=["two_kernels", "mixed_kernel"])
@pytest.mark.parametrize("ctas", [1, 2])
def test_decode_ranges_beyond_staged_ids(runner, ctas, mixed):
    # 2,504 decode blocks: with one CTA at a time no range fits the 1,024 blocks a CTA's
    # range may hold, so the blocks are shared out over three waves of one CTA (chunks of
    # a range's tail go to whichever CTA asks first, in any wave); with two CTAs at a time
    # over two waves.  Rows split across CTAs are merged by the combine kernel.  A prefill
    # chunk rides along, so the metadata kernel's SM split is exercised too.
    spec = wl.StepSpec("long-decode", q_lens=[1, 1, 1, 1, 1, 70], ctx_lens=[8000, 7990, 8016, 7999, 8001, 100],
                       num_blocks=2700, seed=515)
    _run_full_check(runner, spec, ctas=ctas, mixed=mixed)


@pytest.mark.parametrize("mixed", [False, True], ids=["two_kernels", "mixed_kernel"])
def test_many_requests(runner, mixed):
    # 5,000 requests, more than every per-step staging capacity: kv_append's and the decode
    # kernel's shared-memory copies of the step metadata (2,048 requests) fall back to global
    # memory, and the combine kernel's CTA pairs each plan more than one round of rows.
    # Mostly short decode rows (1-3 blocks, so nearly every row is split across pieces),
    # a few empty requests and two prefill chunks.
    rng = np.random.default_rng(9090)
    n = 5000
    q_lens = [1] * n
    ctx = [int(c) for c in rng.integers(0, 48, size=n)]
    for i in rng.choice(n, size=40, replace=False):
        q_lens[i] = 0
    q_lens[1234], ctx[1234] = 70, 19
    q_lens[4321], ctx[4321] = 40, 0
    spec = wl.StepSpec("many-requests", q_lens=q_lens, ctx_lens=ctx, num_blocks=12288, seed=9091)
    _run_full_check(runner, spec, mixed=mixed)


@pytest.mark.parametrize("mixed", [False, True], ids=["two_kernels", "mixed_kernel"])
def test_edge_cases(runner, mixed):
    # an empty request in the middle, decode at positions 0 / 15 / 16 / 31 / 32 / 8192,
    # prefill of 2 rows, a 33-row chunk (two q tiles, one row in the second), a chunk whose
    # cached prefix ends exactly on a 128-key tile boundary and one just before it
    q_lens = [1, 1, 0, 1, 1, 1, 1, 2, 33, 40, 17]
    ctx = [0, 15, 9, 16, 31, 32, 8192, 0, 5, 128, 127]
    spec = wl.StepSpec("edges", q_lens=q_lens, ctx_lens=ctx, num_blocks=1200, seed=4242)
    _run_full_check(runner, spec, mixed=mixed)


def _many_items_spec(seed=0xC0FFEE + 31):
    # 60 short prefill chunks after cached prefixes chosen around 128-key tile edges, plus a
    # few decode rows: several hundred (64-token tile, KV head) work items, so the prefill
    # kernel's CTAs take several items each, one after another
    rng = np.random.default_rng(seed)
    q_lens, ctx = [], []
    for _ in range(60):
        k = int(rng.integers(1, 5))
        ctx.append(int(rng.choice([0, 37, 88, 128 * k - 40, 128 * k - 33, 128 * k - 1, 128 * k + 3])))
        q_lens.append(int(rng.integers(2, 200)))
    q_lens += [1] * 6
    ctx += [int(c) for c in rng.integers(10, 900, size=6)]
    num_blocks = sum(-(-(c + q) // 16) for c, q in zip(ctx, q_lens)) + 64
    return wl.StepSpec("many-prefill-items", q_lens=q_lens, ctx_lens=ctx, num_blocks=num_blocks, seed=seed)


def _tile_shapes(spec):
    # per (request, 64-token tile): the key tiles (of 128) that its two 32-token halves read
    shapes = []
    for q, c in zip(spec.q_lens, spec.ctx_lens):
        if q < 2:
            continue
        for tok0 in range(0, q, 64):
            nt = min(64, q - tok0)
            na, nb = min(32, nt), nt - min(32, nt)
            pa = (c + tok0 + na - 1) // 128 + 1
            pb = (c + tok0 + 32 + nb - 1) // 128 + 1 if nb else 0
            shapes.append((pa, pb))
    return shapes


@pytest.mark.parametrize("mixed", [False, True], ids=["two_kernels", "mixed_kernel"])
def test_prefill_items_in_sequence(runner, mixed):
    # The prefill kernel's CTAs carry their rings, barrier phases and TMEM from one work item
    # to the next: items whose second half is empty, reads the same key tiles as the first,
    # or reads one key tile more, in every order, several per CTA.
    spec = _many_items_spec()
    shapes = _tile_shapes(spec)
    assert len(shapes) * 8 > 2 * 152
    assert sum(pb == 0 for _, pb in shapes) >= 5
    assert sum(pb == pa for pa, pb in shapes) >= 5
    assert sum(pb == pa + 1 for pa, pb in shapes) >= 5
    _run_full_check(runner, spec, mixed=mixed)


@pytest.mark.parametrize("mixed", [False, True], ids=["two_kernels", "mixed_kernel"])
def test_back_to_back_attention_calls_share_workspace(runner, mixed):
    # Three attention calls in a row on one workspace, nothing between them (each into its
    # own output): a call's metadata kernel resets the work counters and rewrites the tile
    # list, so it must not start while the previous call's kernels still read them.  The
    # step has prefill chunks and no decode rows, so the combine kernel has nothing to merge.
    import torch
    spec = wl.StepSpec("prefill-only", q_lens=[1536, 1000, 500], ctx_lens=[1536, 0, 333], num_blocks=512,
                       seed=0xC0FFEE + 33)
    inp = wl.make_inputs(spec)
    step = runner.PagedStep(inp, pool_fill_bits=NAN_BITS, poison_workspace=True, mixed=mixed)
    try:
        step.append()
        nan = int(np.array([NAN_BITS], dtype=np.uint16).view(np.int16)[0])
        outs = [torch.empty_like(step.out) for _ in range(3)]
        for o in outs:
            o.view(torch.int16).fill_(nan)
        torch.cuda.synchronize()
        from continuous_batching_paged_step_gb300 import kvpaged as kp
        for o in outs:
            kp.paged_attention_step(step.pool.handle, step.q, o, step.cu_seqlens_q, step.context_lens,
                                    step.block_tables, step.max_q_len, step.max_context_len, step.softmax_scale,
                                    step.workspace)
        assert step.error() == (0, 0)
        want = oracle.step_reference(inp)
        for i, o in enumerate(outs):
            got = o.float().cpu().numpy().reshape(spec.num_tokens, spec.n_q_heads, spec.head_dim)
            _compare(got, want, what=f"call {i}")
    finally:
        step.close()


def test_chunked_prefill_matches_one_shot(runner):
    # The same 300-token prompt run as chunks of 100, 150 and 50 over three steps through
    # the pool equals one-shot causal prefill (chunked prefill, page "Continuous Batching
    # 深入实现", section "第三层：Chunked Prefill").
    import torch
    from continuous_batching_paged_step_gb300 import kvpaged as kp
    full = wl.StepSpec("prompt300", q_lens=[300], ctx_lens=[0], num_blocks=64, seed=99)
    inp = wl.make_inputs(full)
    want = oracle.step_reference(inp)
    step = runner.PagedStep(inp, pool_fill_bits=NAN_BITS)
    try:
        done = 0
        for C in (100, 150, 50):
            rows = slice(done, done + C)
            dev = step.device
            q = step.q[rows].contiguous()
            out = torch.zeros_like(q)
            cu = torch.tensor([0, C], dtype=torch.int32, device=dev)
            ctx = torch.tensor([done], dtype=torch.int32, device=dev)
            kp.kv_append(step.pool.handle, step.k_new[rows].contiguous(), step.v_new[rows].contiguous(), cu, ctx,
                         step.block_tables)
            ws = torch.empty(kp.paged_attention_workspace_size(step.pool.handle, 1, C, done), dtype=torch.uint8,
                             device=dev)
            kp.paged_attention_step(step.pool.handle, q, out, cu, ctx, step.block_tables, C, done,
                                    step.softmax_scale, ws)
            got = out.float().cpu().numpy().reshape(C, 32, 128)
            _compare(got, want[rows], what=f"chunk at {done}")
            done += C
        assert step.error() == (0, 0)
    finally:
        step.close()


def _sample_rows(spec, rng, per_req=3):
    cu = np.concatenate([[0], np.cumsum(spec.q_lens)])
    rows = []
    for r, ql in enumerate(spec.q_lens):
        if ql == 0:
            continue
        if ql == 1:
            rows.append(cu[r])
        else:
            pick = {0, ql - 1, 31, 32, ql // 2} | set(rng.integers(0, ql, size=per_req).tolist())
            rows += [cu[r] + j for j in sorted(pick) if j < ql]
    return np.array(sorted(set(int(x) for x in rows)))


@pytest.mark.parametrize("mixed", [False, True], ids=["two_kernels", "mixed_kernel"])
@pytest.mark.parametrize("name", ["mixed", "decode", "chunked"])
def test_full_size_configs_sampled(runner, name, mixed):
    spec = wl.CONFIGS[name]()
    inp = wl.make_inputs(spec)
    step = runner.PagedStep(inp, mixed=mixed)
    try:
        step.run()
        assert step.error() == (0, 0)
        rng = np.random.default_rng(5)
        rows = _sample_rows(spec, rng)
        if name == "decode":
            rows = rows[rng.permutation(len(rows))[:48]]
        want = oracle.step_reference(inp, rows=rows)
        _compare(step.out_f32(), want, rows=rows, what=name)
        # kv_append bit-exact at the sampled rows: read each row back through the table
        k, v = ph.pool_bits(step)
        cu = inp.cu_seqlens_q
        for i in rows[:64]:
            r = int(np.searchsorted(cu, i, side="right") - 1)
            p = int(inp.context_lens[r] + i - cu[r])
            b, off, _ = oracle.physical_slot(inp.block_tables[r], p)
            assert np.array_equal(k[b, :, off, :].reshape(-1), inp.k_new[i])
            assert np.array_equal(v[b, :, off, :].reshape(-1), inp.v_new[i])
    finally:
        step.close()


@pytest.mark.parametrize("case", range(12))
def test_random_step_shapes(runner, case):
    # Random packed steps: empty requests, decode rows and prefill chunks in any order,
    # contexts from 0 to ~2,000 (log-uniform, so short and block-boundary ones are common),
    # a random decode CTA cap; the whole output and the pool are checked.
    rng = np.random.default_rng(9000 + case)
    R = int(rng.integers(1, 24))
    q_lens, ctx_lens = [], []
    for _ in range(R):
        kind = rng.random()
        q = 0 if kind < 0.08 else 1 if kind < 0.65 else int(rng.integers(2, 160))
        c = int(np.exp(rng.uniform(0, np.log(2100)))) - 1 if rng.random() < 0.9 else int(rng.integers(0, 3)) * 16
        q_lens.append(q)
        ctx_lens.append(c)
    need = sum(-(-(c + q) // 16) for c, q in zip(ctx_lens, q_lens))
    spec = wl.StepSpec(f"random-{case}", q_lens=q_lens, ctx_lens=ctx_lens, num_blocks=need + int(rng.integers(1, 64)),
                       seed=7000 + case)
    if spec.num_tokens == 0:
        spec.q_lens[0] = 1
    ctas = [0, 1, 3, 16][case % 4]
    _run_full_check(runner, spec, ctas=ctas, mixed=case % 3 == 1)
