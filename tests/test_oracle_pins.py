"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: values printed on the
pages (the mask grids), closed forms, library routines for special cases, and
invariants the pages state (packing equals running each request alone; chunked prefill
equals one-shot prefill).  They are chosen so that a dropped scale, a wrong GQA head
map, an off-by-one in the causal test, a context length that counts this step's tokens,
or a transposed operand each fail at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from continuous_batching_paged_step_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_bf16(rng, shape):
    return wl.f32_to_bf16_bits(rng.standard_normal(int(np.prod(shape)), dtype=np.float32)).reshape(shape)


def _bf16_exact(values):
    """bf16 bits of float values that are exactly representable (checked)."""
    f = np.asarray(values, dtype=np.float32)
    bits = (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    assert np.array_equal(wl.bf16_bits_to_f32(bits), f)
    return bits


# ------------------------------------------------------------------ address mapping

def test_address_mapping_closed_form():
    # Page "连续批处理与 PagedAttention 原理", section "block table 与地址映射":
    # logical block p // 16, physical block b from the table, slot b * 16 + p % 16.
    table = [7, 2, 9]
    expect = {0: (7, 0, 112), 15: (7, 15, 127), 16: (2, 0, 32), 31: (2, 15, 47),
              32: (9, 0, 144), 40: (9, 8, 152), 47: (9, 15, 159)}
    for p, want in expect.items():
        assert oracle.physical_slot(table, p) == want


def test_cache_write_hits_mapped_slots_and_nothing_else():
    n_kv, d, nb = 2, 8, 6
    sentinel = 0x3F80  # bf16 1.0, a finite value
    kc = np.full((nb, n_kv, 16, d), sentinel, np.uint16)
    vc = np.full((nb, n_kv, 16, d), sentinel, np.uint16)
    # one request: 5 tokens cached, 30 new -> positions 5..34 over blocks [5, 0, 3]
    T = 30
    k_new = (np.arange(T * n_kv * d, dtype=np.uint32) % 50000 + 1).astype(np.uint16).reshape(T, n_kv * d)
    v_new = (k_new.astype(np.uint32) + 7).astype(np.uint16)
    cu = np.array([0, T], np.int32)
    ctx = np.array([5], np.int32)
    tables = np.array([[5, 0, 3]], np.int32)
    k2, v2 = oracle.reference_cache_write(kc, vc, k_new, v_new, cu, ctx, tables, n_kv, d)
    # hand-checked destinations: row 0 is position 5 -> block 5 offset 5; row 11 is
    # position 16 -> block 0 offset 0; row 29 is position 34 -> block 3 offset 2
    for row, (b, off) in {0: (5, 5), 10: (5, 15), 11: (0, 0), 26: (0, 15), 27: (3, 0), 29: (3, 2)}.items():
        for h in range(n_kv):
            assert np.array_equal(k2[b, h, off], k_new[row, h * d:(h + 1) * d])
            assert np.array_equal(v2[b, h, off], v_new[row, h * d:(h + 1) * d])
    changed = np.any(k2 != sentinel, axis=-1)
    assert changed.sum() == T * n_kv
    assert not changed[[1, 2, 4]].any()          # blocks outside the table untouched
    assert not changed[5, :, :5].any()           # the 5 cached slots are not rewritten
    assert not changed[3, :, 3:].any()           # tail of the last block untouched


def test_reverse_gather_identity_random_tables():
    rng = np.random.default_rng(5)
    n_kv, d, nb = 2, 16, 40
    ctx = [0, 17, 31, 3]
    ql = [9, 1, 16, 20]
    need = [-(-(c + q) // 16) for c, q in zip(ctx, ql)]
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((4, max(need)), -1, np.int32)
    o = 0
    for r in range(4):
        tables[r, :need[r]] = perm[o:o + need[r]]
        o += need[r]
    kc = np.zeros((nb, n_kv, 16, d), np.uint16)
    vc = np.zeros_like(kc)
    # first write each request's cached prefix, then this step's rows
    prior_k = [_rand_bf16(rng, (c, n_kv * d)) for c in ctx]
    prior_v = [_rand_bf16(rng, (c, n_kv * d)) for c in ctx]
    cu0 = np.concatenate([[0], np.cumsum(ctx)]).astype(np.int32)
    kc, vc = oracle.reference_cache_write(kc, vc, np.concatenate(prior_k), np.concatenate(prior_v),
                                          cu0, np.zeros(4, np.int32), tables, n_kv, d)
    T = sum(ql)
    k_new, v_new = _rand_bf16(rng, (T, n_kv * d)), _rand_bf16(rng, (T, n_kv * d))
    cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    kc, vc = oracle.reference_cache_write(kc, vc, k_new, v_new, cu, np.array(ctx, np.int32), tables, n_kv, d)
    for r in range(4):
        want_k = np.concatenate([prior_k[r], k_new[cu[r]:cu[r + 1]]])
        want_v = np.concatenate([prior_v[r], v_new[cu[r]:cu[r + 1]]])
        assert np.array_equal(oracle.gather_request(kc, tables[r], ctx[r] + ql[r]), want_k)
        assert np.array_equal(oracle.gather_request(vc, tables[r], ctx[r] + ql[r]), want_v)


def test_shared_prefix_blocks_figure_11_4():
    # Page "11.2 连续批处理与 PagedAttention", section 11.2.3, Figure 11-4: A holds 50
    # tokens on blocks 1, 4, 7, 2; B holds 40 on blocks 1, 4, 8; blocks 1 and 4 are full
    # and shared read-only.  B's own tokens start at position 32, in block 8.
    n_kv, d, nb = 1, 4, 10
    rng = np.random.default_rng(11)
    kc = np.zeros((nb, n_kv, 16, d), np.uint16)
    vc = np.zeros_like(kc)
    ka, va = _rand_bf16(rng, (50, d)), _rand_bf16(rng, (50, d))
    kc, vc = oracle.reference_cache_write(kc, vc, ka, va, np.array([0, 50], np.int32),
                                          np.array([0], np.int32), np.array([[1, 4, 7, 2]], np.int32), n_kv, d)
    kb, vb = _rand_bf16(rng, (8, d)), _rand_bf16(rng, (8, d))
    before = kc.copy()
    kc, vc = oracle.reference_cache_write(kc, vc, kb, vb, np.array([0, 8], np.int32),
                                          np.array([32], np.int32), np.array([[1, 4, 8]], np.int32), n_kv, d)
    assert np.array_equal(kc[[1, 4, 7, 2]], before[[1, 4, 7, 2]])   # A's blocks untouched by B
    gb = oracle.gather_request(kc, [1, 4, 8], 40)
    assert np.array_equal(gb[:32], ka[:32]) and np.array_equal(gb[32:], kb)
    used = np.any(kc != 0, axis=-1)[:, 0, :].sum(axis=1)
    assert used[1] == 16 and used[4] == 16 and used[7] == 16    # full blocks
    assert used[2] == 50 - 48 and used[8] == 40 - 32            # partial tails


def test_prefix_sharing_counts_full_blocks_only():
    # Page "11.2", section 11.2.4: with 2,010 shared tokens and 16-token blocks only full
    # blocks can be shared: 125 blocks = 2,000 tokens.
    shared_tokens = 2010
    full_blocks = shared_tokens // 16
    assert full_blocks == 125 and full_blocks * 16 == 2000
    # the last shared position that lies in a full block maps inside logical block 124
    assert oracle.physical_slot(list(range(200)), 1999)[0] == 124
    assert oracle.physical_slot(list(range(200)), 2000)[0] == 125


# ------------------------------------------------------------------------ the mask

def _read_grid(name):
    seqs, keys, rows = None, None, []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.rstrip("\n")
            if not line or line.startswith("%"):
                continue
            if line.startswith("seqs:"):
                seqs = [tuple(t.split(":")) for t in line.split()[1:]]
                seqs = [(lab, int(n), int(c)) for lab, n, c in seqs]
            elif line.startswith("keys:"):
                keys = line[len("keys:"):].strip()
            else:
                lab, pos, cells = line.split(" ", 2)
                rows.append((lab, int(pos[1:]), cells))
    return seqs, keys, rows


def _format_cells(values, key_seq, n_cached):
    out = []
    for j, v in enumerate(values):
        if n_cached > 0 and j == n_cached:
            out.append(" | ")
        elif j > 0 and key_seq[j] != key_seq[j - 1]:
            out.append(" ")
        out.append(v)
    return "".join(out)


@pytest.mark.parametrize("name", ["p1_mask_step1.txt", "p1_mask_step7.txt"])
def test_mask_grids_printed_on_page(name):
    seqs, keys, rows = _read_grid(name)
    labels = [s[0] for s in seqs]
    q_lens = [s[1] for s in seqs]
    ctx = [s[2] for s in seqs]
    q_seq, q_pos, key_seq, key_pos = oracle.packed_key_layout(q_lens, ctx)
    allowed = oracle.block_diagonal_causal_mask(q_seq, q_pos, key_seq, key_pos)
    n_cached = sum(ctx)
    assert _format_cells([labels[s] for s in key_seq], key_seq, n_cached) == keys
    assert len(rows) == len(q_seq)
    for i, (lab, pos, cells) in enumerate(rows):
        assert (lab, pos) == (labels[q_seq[i]], q_pos[i])
        got = _format_cells(["#" if a else "." for a in allowed[i]], key_seq, n_cached)
        assert got == cells, f"row {lab} p{pos}"


def test_three_request_score_shapes():
    # Page "11.2", section 11.2.2: R1 prefills 5 tokens (scores [5, 5], causal), R2
    # decodes with 7 cached (scores [1, 8]), R3 decodes with 3 cached (scores [1, 4]).
    q_seq, q_pos, key_seq, key_pos = oracle.packed_key_layout([5, 1, 1], [0, 7, 3])
    allowed = oracle.block_diagonal_causal_mask(q_seq, q_pos, key_seq, key_pos)
    assert allowed.shape == (7, 0 + 7 + 3 + 7)
    assert allowed.sum(axis=1).tolist() == [1, 2, 3, 4, 5, 8, 4]
    # R1's visible keys form a lower-triangular 5x5 block
    r1_cols = [j for j, s in enumerate(key_seq) if s == 0]
    assert np.array_equal(allowed[:5][:, r1_cols], np.tril(np.ones((5, 5), bool)))


# -------------------------------------------------------------------- the softmax

def test_softmax_rows_sum_to_one_and_masked_weights_are_zero():
    rng = np.random.default_rng(3)
    s = rng.standard_normal((50, 37)) * 30
    s[:, 20:] = -np.inf
    s[:, 0] = rng.standard_normal(50)
    w = oracle.softmax_weights(s)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-12, rtol=0)
    assert np.all(w[:, 20:] == 0.0)
    assert np.all(w >= 0)


def test_two_key_weights_are_logistic():
    # With two keys the softmax weight of the first is the logistic of the score gap.
    s1, s2 = 0.75, -1.25
    w = oracle.softmax_weights(np.array([[s1, s2]]))
    assert abs(w[0, 0] - 1.0 / (1.0 + math.exp(s2 - s1))) < 1e-15


def _single_request(q, k_hist, v_hist, ctx, n_q, n_kv, d):
    T = q.shape[0]
    return oracle.attention_reference(q, [k_hist], [v_hist], np.array([0, T], np.int32),
                                      np.array([ctx], np.int32), n_q, n_kv, d)


def test_single_key_context_returns_its_value():
    rng = np.random.default_rng(4)
    n_q, n_kv, d = 32, 8, 128
    q = _rand_bf16(rng, (1, n_q * d))
    k = _rand_bf16(rng, (1, n_kv * d))
    v = _rand_bf16(rng, (1, n_kv * d))
    out = _single_request(q, k, v, 0, n_q, n_kv, d)
    vv = oracle.bf16_to_f64(v).reshape(n_kv, d)
    for h in range(n_q):
        assert np.array_equal(out[0, h], vv[h // 4])


def test_constant_values_give_that_constant():
    rng = np.random.default_rng(6)
    n_q, n_kv, d, ctx, T = 8, 2, 16, 21, 6
    q = _rand_bf16(rng, (T, n_q * d))
    k = _rand_bf16(rng, (ctx + T, n_kv * d))
    c = _bf16_exact(np.arange(n_kv * d, dtype=np.float32) / 8 - 3)
    v = np.tile(c, (ctx + T, 1))
    out = _single_request(q, k, v, ctx, n_q, n_kv, d)
    want = oracle.bf16_to_f64(c).reshape(n_kv, d)
    for h in range(n_q):
        assert np.allclose(out[:, h], want[h // 4][None, :], atol=1e-12, rtol=0)


def test_hand_computed_two_token_example():
    # One head, d = 2: keys (1, 0) and (0, 1), values (2, 0) and (0, 4), query (2, 0).
    # Scores are 2/sqrt(2) and 0, so the first weight is the logistic of sqrt(2).
    q = _bf16_exact([[2.0, 0.0]])
    k = _bf16_exact([[1.0, 0.0], [0.0, 1.0]])
    v = _bf16_exact([[2.0, 0.0], [0.0, 4.0]])
    out = oracle.attention_reference(q, [k], [v], np.array([0, 1], np.int32),
                                     np.array([1], np.int32), 1, 1, 2)
    w1 = 1.0 / (1.0 + math.exp(-math.sqrt(2.0)))
    assert np.allclose(out[0, 0], [2.0 * w1, 4.0 * (1.0 - w1)], atol=1e-15, rtol=0)


# ------------------------------------------------ against library routines (torch)

def _sdpa(qf, kf, vf, causal, n_q, n_kv):
    """torch scaled_dot_product_attention in fp64 with KV heads repeated to query heads."""
    g = n_q // n_kv
    Q = torch.from_numpy(qf).permute(1, 0, 2)                  # [H, L, d]
    K = torch.from_numpy(kf).permute(1, 0, 2).repeat_interleave(g, dim=0)
    V = torch.from_numpy(vf).permute(1, 0, 2).repeat_interleave(g, dim=0)
    o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=causal)
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("n_q,n_kv,d,T", [(32, 8, 128, 21), (4, 2, 16, 40), (6, 3, 8, 1)])
def test_prefill_without_cache_is_causal_sdpa(n_q, n_kv, d, T):
    rng = np.random.default_rng(T + d)
    q = _rand_bf16(rng, (T, n_q * d))
    k = _rand_bf16(rng, (T, n_kv * d))
    v = _rand_bf16(rng, (T, n_kv * d))
    out = _single_request(q, k, v, 0, n_q, n_kv, d)
    f = lambda a, h: oracle.bf16_to_f64(a).reshape(-1, h, d)
    want = _sdpa(f(q, n_q), f(k, n_kv), f(v, n_kv), True, n_q, n_kv)
    assert np.allclose(out, want, atol=1e-12, rtol=0)


def test_decode_row_sees_whole_history_as_sdpa():
    # The decode formula on the k4i.top page ("与 KV cache 的关系"): one query row against
    # [K_cache; k_t] and [V_cache; v_t], i.e. unmasked attention over ctx + 1 keys.
    rng = np.random.default_rng(8)
    n_q, n_kv, d, ctx = 32, 8, 128, 45
    q = _rand_bf16(rng, (1, n_q * d))
    k = _rand_bf16(rng, (ctx + 1, n_kv * d))
    v = _rand_bf16(rng, (ctx + 1, n_kv * d))
    out = _single_request(q, k, v, ctx, n_q, n_kv, d)
    f = lambda a, h: oracle.bf16_to_f64(a).reshape(-1, h, d)
    want = _sdpa(f(q, n_q), f(k, n_kv), f(v, n_kv), False, n_q, n_kv)
    assert np.allclose(out, want, atol=1e-12, rtol=0)
    # a history that (wrongly) stopped before this step's own key differs
    short = _sdpa(f(q, n_q), f(k[:-1], n_kv), f(v[:-1], n_kv), False, n_q, n_kv)
    assert np.abs(out - short).max() > 1e-3


def test_packed_dense_mask_equals_separate_requests():
    # Packing equals running every request alone (k4i.top page, "为什么 packed forward
    # 等价"); shapes of the 3-request example on page "11.2", section 11.2.2.
    inp = wl.make_inputs(wl.tiny_p5_step())
    spec = inp.spec
    ks, vs = oracle.request_histories(inp)
    sep = oracle.step_reference(inp)
    dense = oracle.attention_dense_mask(inp.q, inp.k_prior, inp.v_prior, inp.k_new, inp.v_new,
                                        inp.cu_seqlens_q, inp.context_lens,
                                        spec.n_q_heads, spec.n_kv_heads, spec.head_dim)
    assert np.allclose(dense, sep, atol=1e-12, rtol=0)
    d = spec.head_dim
    f = lambda a, h: oracle.bf16_to_f64(a).reshape(-1, h, d)
    for r in range(spec.num_reqs):
        s, e = inp.cu_seqlens_q[r], inp.cu_seqlens_q[r + 1]
        # each request alone: its rows are the last rows of a causal prefill over its
        # whole history, so run causal SDPA on (history queries = zero-padded) and keep
        # the tail -- valid because causal rows never look right.
        N = ks[r].shape[0]
        qfull = np.zeros((N, spec.n_q_heads, d))
        qfull[N - (e - s):] = f(inp.q[s:e], spec.n_q_heads)
        want = _sdpa(qfull, f(ks[r], spec.n_kv_heads), f(vs[r], spec.n_kv_heads), True,
                     spec.n_q_heads, spec.n_kv_heads)[N - (e - s):]
        assert np.allclose(sep[s:e], want, atol=1e-12, rtol=0)


def test_chunked_prefill_equals_one_shot():
    # Chunked prefill (page "Continuous Batching 深入实现", section "第三层：Chunked
    # Prefill"): chunk k attends to the KV that earlier chunks wrote plus its own rows.
    rng = np.random.default_rng(12)
    n_q, n_kv, d = 8, 2, 32
    N = 45
    q = _rand_bf16(rng, (N, n_q * d))
    k = _rand_bf16(rng, (N, n_kv * d))
    v = _rand_bf16(rng, (N, n_kv * d))
    one_shot = _single_request(q, k, v, 0, n_q, n_kv, d)
    table = np.array([[3, 0, 2]], np.int32)
    kc = np.zeros((4, n_kv, 16, d), np.uint16)
    vc = np.zeros_like(kc)
    done = 0
    for C in (13, 20, 12):
        cu = np.array([0, C], np.int32)
        ctx = np.array([done], np.int32)
        kc, vc = oracle.reference_cache_write(kc, vc, k[done:done + C], v[done:done + C], cu, ctx, table, n_kv, d)
        kh = oracle.gather_request(kc, table[0], done + C)
        vh = oracle.gather_request(vc, table[0], done + C)
        part = oracle.attention_reference(q[done:done + C], [kh], [vh], cu, ctx, n_q, n_kv, d)
        assert np.allclose(part, one_shot[done:done + C], atol=1e-12, rtol=0)
        done += C


def test_invariant_to_request_order_and_block_placement():
    spec = wl.small_mixed_step(n_decode=3, chunks=((20, 9), (5, 0)), ctx_range=(1, 40), num_blocks=64)
    inp = wl.make_inputs(spec)
    base = oracle.step_reference(inp)
    # reverse the request order in the pack
    order = list(range(spec.num_reqs))[::-1]
    q_rows, cu = [], [0]
    for r in order:
        s, e = inp.cu_seqlens_q[r], inp.cu_seqlens_q[r + 1]
        q_rows.append(np.arange(s, e))
        cu.append(cu[-1] + e - s)
    idx = np.concatenate(q_rows)
    ks, vs = oracle.request_histories(inp)
    out = oracle.attention_reference(inp.q[idx], [ks[r] for r in order], [vs[r] for r in order],
                                     np.array(cu, np.int32), inp.context_lens[order],
                                     spec.n_q_heads, spec.n_kv_heads, spec.head_dim)
    assert np.array_equal(out, base[idx])
    # physical placement: histories read back through two different block tables agree
    d, n_kv = spec.head_dim, spec.n_kv_heads
    for seed in (1, 2):
        perm = np.random.default_rng(seed).permutation(spec.num_blocks).astype(np.int32)
        tables = np.full_like(inp.block_tables, -1)
        o = 0
        for r in range(spec.num_reqs):
            n = spec.blocks_needed(r)
            tables[r, :n] = perm[o:o + n]
            o += n
        kc = np.zeros((spec.num_blocks, n_kv, 16, d), np.uint16)
        vc = np.zeros_like(kc)
        N = [spec.ctx_lens[r] + spec.q_lens[r] for r in range(spec.num_reqs)]
        cuh = np.concatenate([[0], np.cumsum(N)]).astype(np.int32)
        kc, vc = oracle.reference_cache_write(kc, vc, np.concatenate(ks), np.concatenate(vs), cuh,
                                              np.zeros(spec.num_reqs, np.int32), tables, n_kv, d)
        kh = [oracle.gather_request(kc, tables[r], N[r]) for r in range(spec.num_reqs)]
        vh = [oracle.gather_request(vc, tables[r], N[r]) for r in range(spec.num_reqs)]
        out = oracle.attention_reference(inp.q, kh, vh, inp.cu_seqlens_q, inp.context_lens,
                                         spec.n_q_heads, n_kv, d)
        assert np.array_equal(out, base)


def test_empty_request_produces_no_rows():
    rng = np.random.default_rng(13)
    n_q, n_kv, d = 4, 2, 8
    q = _rand_bf16(rng, (3, n_q * d))
    k0, v0 = _rand_bf16(rng, (5, n_kv * d)), _rand_bf16(rng, (5, n_kv * d))
    k1, v1 = _rand_bf16(rng, (4, n_kv * d)), _rand_bf16(rng, (4, n_kv * d))
    cu = np.array([0, 0, 3], np.int32)          # request 0 brings no rows this step
    out = oracle.attention_reference(q, [k0, k1], [v0, v1], cu, np.array([5, 1], np.int32), n_q, n_kv, d)
    alone = oracle.attention_reference(q, [k1], [v1], np.array([0, 3], np.int32),
                                       np.array([1], np.int32), n_q, n_kv, d)
    assert np.array_equal(out, alone)
