"""Shared pieces of the GPU parity checks and of the needle / late-peak checks (test
infrastructure).

The comparison rule is the parity bar for bf16 attention outputs: max-abs <= 2e-2 and
mean-abs <= 2e-3 against the fp64 oracle.  `compare_rows` picks the packed rows a check
compares: every decode row, and in each prefill chunk its first and last rows, the rows
on both sides of every 32- and 64-token q-tile boundary up to the 128th, and rows spread
evenly over the rest.  `mutated_reference` is the oracle run on a history with one block
of keys removed or repeated: the check must tell it apart from the true output.
`oracle_pool` is the oracle's cache write of a whole step into a sentinel-filled pool
(every request's cached tokens first, then the step's new rows).
"""
import numpy as np

import oracle

MAX_ABS, MEAN_ABS = 2e-2, 2e-3


def errors(got, want):
    err = np.abs(np.asarray(got, dtype=np.float64) - want)
    return float(err.max()), float(err.mean())


def within_tolerance(got, want):
    mx, mn = errors(got, want)
    return mx <= MAX_ABS and mn <= MEAN_ABS


def compare_rows(inp, spread: int = 97):
    cu = inp.cu_seqlens_q
    rows = []
    for r in range(len(inp.context_lens)):
        a, b = int(cu[r]), int(cu[r + 1])
        if b - a <= 40:
            rows += list(range(a, b))
            continue
        near = [0, 1, 31, 32, 33, 63, 64, 65, 95, 96, 127, 128]
        rows += [a + j for j in near if a + j < b] + [b - 2, b - 1] + list(range(a, b, spread))
    return np.array(sorted(set(rows)), dtype=np.int64)


def rows_of_request(inp, r, rows):
    cu = inp.cu_seqlens_q
    return [int(i) for i in rows if cu[r] <= i < cu[r + 1]]


def mutated_reference(inp, r, block, mode, rows):
    """Oracle output of request r's listed rows when its history loses (mode 'drop') or
    repeats ('dup') the cached keys of logical block `block`."""
    spec = inp.spec
    ks, vs = oracle.request_histories(inp, {r})
    c = int(inp.context_lens[r])
    lo, hi = block * spec.block_size, min((block + 1) * spec.block_size, c)
    idx = np.arange(ks[r].shape[0])
    if mode == "drop":
        keep = np.concatenate([idx[:lo], idx[hi:]])
    else:
        keep = np.concatenate([idx[:hi], idx[lo:hi], idx[hi:]])
    k2, v2 = [None] * len(ks), [None] * len(vs)
    k2[r], v2[r] = ks[r][keep], vs[r][keep]
    ctx2 = np.array(inp.context_lens, copy=True)
    ctx2[r] = c + (keep.shape[0] - idx.shape[0])
    return oracle.attention_reference(inp.q, k2, v2, inp.cu_seqlens_q, ctx2, spec.n_q_heads, spec.n_kv_heads,
                                      spec.head_dim, rows=rows)


def oracle_pool(inp, fill_bits):
    spec = inp.spec
    shape = (spec.num_blocks, spec.n_kv_heads, spec.block_size, spec.head_dim)
    kc = np.full(shape, fill_bits, np.uint16)
    vc = np.full(shape, fill_bits, np.uint16)
    ctx = np.asarray(inp.context_lens)
    cu0 = np.concatenate([[0], np.cumsum(ctx)]).astype(np.int32)
    kp_ = [k for k in inp.k_prior if k is not None and k.shape[0]]
    vp_ = [v for v in inp.v_prior if v is not None and v.shape[0]]
    if kp_:
        kc, vc = oracle.reference_cache_write(kc, vc, np.concatenate(kp_), np.concatenate(vp_), cu0,
                                              np.zeros_like(ctx), inp.block_tables, spec.n_kv_heads, spec.head_dim)
    return oracle.reference_cache_write(kc, vc, inp.k_new, inp.v_new, inp.cu_seqlens_q, inp.context_lens,
                                        inp.block_tables, spec.n_kv_heads, spec.head_dim)


def pool_bits(step):
    import torch
    k = step.pool.k_cache.view(torch.int16).cpu().numpy().view(np.uint16)
    v = step.pool.v_cache.view(torch.int16).cpu().numpy().view(np.uint16)
    return k, v
