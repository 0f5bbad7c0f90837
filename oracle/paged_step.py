"""CPU oracle for one packed continuous-batching step (kv_append + paged attention).

TEST INFRASTRUCTURE ONLY.  This module is the slow, plain, fp64 statement of what the
GPU path computes.  Only the test suite, the smoke check and the CPU-baseline leg of the
benchmark may import it; the product path never does.  It shares no code with the CUDA
library: it imports nothing from the package except, in callers, the seeded input
generator.

What is computed, and where the pages define it:

* Block-table address mapping (page "连续批处理与 PagedAttention 原理", section
  "block table 与地址映射"): logical position p of a request lies in logical block
  p // 16; that entry of the request's block table names physical block b; the physical
  token slot is b * 16 + p % 16.  The pool stores each block as [n_kv][16][d] (one
  (block, head) tile is contiguous), so token slot (b, p % 16) of head h starts at
  element ((b * n_kv + h) * 16 + p % 16) * d.

* Appending this step's K/V (page "Continuous Batching" on k4i.top, section "一个完整的
  mixed iteration", and page "11.2 连续批处理与 PagedAttention", section 11.2.2): row j of
  request r holds position ctx_r + j, where ctx_r counts the tokens cached before this
  step (page "同时服务多位用户：连续批处理如何保持 LLM 推理高效", section "完整实现", the
  `_ragged_step` routine numbers a new token as its sequence's cached length plus its
  index).  The oracle writes it gather-free, one token at a time.

* Attention (k4i.top page, sections "防止跨请求 attention" (the mask M_ij) and "为什么
  packed forward 等价" (the visible set S(i)); decode formula in "与 KV cache 的关系"):
  the row at position P of request r attends to positions 0..P of r only, with weights
  softmax(q . k / sqrt(d)).  Packing does not change the result, so the oracle runs each
  request on its own contiguous K/V ("attention_reference") and never reads the pool.
  "attention_dense_mask" is the packed brute-force form with the explicit additive
  block-diagonal causal mask over [cached keys | new keys], as in the ragged-batching
  routine of the "同时服务多位用户" page; the tests require the two to agree.

* GQA: 32 query heads over 8 KV heads; query head h reads KV head h // (n_q / n_kv).
  The pages name GQA with 8 KV heads of 128 dims (page "Continuous Batching", section
  "为什么 decode 是 bandwidth-bound"; page "11.2", section 11.2.2 shows W_K as
  [4096, 1024]) but do not give the head map; contiguous groups are the plain reading.

bf16 values arrive as uint16 bit patterns and are widened to fp64 exactly.
"""
from __future__ import annotations

import numpy as np

BLOCK_SIZE = 16


# ----------------------------------------------------------------------------- helpers

def bf16_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns: bf16 is the top half of an IEEE float32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32)
    return (b << np.uint32(16)).view(np.float32).astype(np.float64)


def physical_slot(table_row, p: int, block_size: int = BLOCK_SIZE):
    """Address mapping of a logical position p through one request's block table.

    Returns (b, offset, slot) with b = table_row[p // block_size],
    offset = p % block_size and slot = b * block_size + offset.
    """
    b = int(table_row[p // block_size])
    off = p % block_size
    return b, off, b * block_size + off


# ----------------------------------------------------------------------- cache write

def reference_cache_write(k_cache, v_cache, k_new, v_new, cu_seqlens_q, context_lens,
                          block_tables, n_kv_heads: int, head_dim: int,
                          block_size: int = BLOCK_SIZE):
    """Return copies of the pools with this step's K/V rows written in.

    k_cache, v_cache: uint16 [num_blocks, n_kv, block_size, d]
    k_new, v_new:     uint16 [T, n_kv * d]
    Each token is copied bit for bit: for request r, row j, head h the position is
    p = ctx_r + j and the destination is pool[b, h, p % block_size, :] with
    b = table[r][p // block_size].
    """
    kc = np.array(k_cache, dtype=np.uint16, copy=True)
    vc = np.array(v_cache, dtype=np.uint16, copy=True)
    R = len(context_lens)
    for r in range(R):
        start, end = int(cu_seqlens_q[r]), int(cu_seqlens_q[r + 1])
        for j in range(end - start):
            i = start + j
            p = int(context_lens[r]) + j
            b, off, _ = physical_slot(block_tables[r], p, block_size)
            for h in range(n_kv_heads):
                cols = slice(h * head_dim, (h + 1) * head_dim)
                kc[b, h, off, :] = k_new[i, cols]
                vc[b, h, off, :] = v_new[i, cols]
    return kc, vc


def gather_request(cache, table_row, n_tokens: int, block_size: int = BLOCK_SIZE):
    """Read positions 0..n_tokens-1 of one request back out of a pool.

    Returns uint16 [n_tokens, n_kv * d] in the packed row layout.
    """
    num_blocks, n_kv, bs, d = cache.shape
    out = np.empty((n_tokens, n_kv * d), dtype=np.uint16)
    for p in range(n_tokens):
        b, off, _ = physical_slot(table_row, p, block_size)
        for h in range(n_kv):
            out[p, h * d:(h + 1) * d] = cache[b, h, off, :]
    return out


# ------------------------------------------------------------------------- attention

def softmax_weights(scores: np.ndarray) -> np.ndarray:
    """Row-wise softmax of fp64 scores; -inf entries get weight 0."""
    m = np.max(scores, axis=-1, keepdims=True)
    e = np.exp(scores - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attention_reference(q, k_seqs, v_seqs, cu_seqlens_q, context_lens, n_q_heads: int,
                        n_kv_heads: int, head_dim: int, softmax_scale=None, rows=None):
    """Per-request causal attention on contiguous K/V, in fp64.

    q:       uint16 [T, n_q * d]  (this step's packed query rows)
    k_seqs:  per request uint16 [ctx_r + q_r, n_kv * d]: the request's whole K history
             (cached tokens followed by this step's new tokens), contiguous
    v_seqs:  same for V
    rows:    optional iterable of packed row indices to compute (others stay NaN)
    Returns fp64 [T, n_q, d].
    """
    T = q.shape[0]
    d = head_dim
    group = n_q_heads // n_kv_heads
    scale = (1.0 / np.sqrt(float(d))) if softmax_scale is None else float(softmax_scale)
    out = np.full((T, n_q_heads, d), np.nan, dtype=np.float64)
    wanted = None if rows is None else set(int(i) for i in rows)
    R = len(context_lens)
    for r in range(R):
        start, end = int(cu_seqlens_q[r]), int(cu_seqlens_q[r + 1])
        if end == start:
            continue
        js = [j for j in range(end - start) if wanted is None or (start + j) in wanted]
        if not js:
            continue
        ctx = int(context_lens[r])
        K = bf16_to_f64(k_seqs[r]).reshape(-1, n_kv_heads, d)
        V = bf16_to_f64(v_seqs[r]).reshape(-1, n_kv_heads, d)
        if K.shape[0] != ctx + (end - start):
            raise ValueError(f"request {r}: K history has {K.shape[0]} rows, "
                             f"expected {ctx + end - start}")
        Q = bf16_to_f64(q[[start + j for j in js]]).reshape(len(js), n_q_heads, d)
        pos = np.array([ctx + j for j in js])
        key_pos = np.arange(K.shape[0])
        visible = key_pos[None, :] <= pos[:, None]          # [rows, keys]
        for h in range(n_q_heads):
            kvh = h // group
            s = (Q[:, h, :] @ K[:, kvh, :].T) * scale       # [rows, keys]
            s = np.where(visible, s, -np.inf)
            w = softmax_weights(s)
            out[[start + j for j in js], h, :] = w @ V[:, kvh, :]
    return out


def block_diagonal_causal_mask(q_seq, q_pos, key_seq, key_pos) -> np.ndarray:
    """allowed[i, j] is True iff key j belongs to the same request as query i and its
    position is not after the query's position (the mask M_ij)."""
    q_seq, q_pos = np.asarray(q_seq), np.asarray(q_pos)
    key_seq, key_pos = np.asarray(key_seq), np.asarray(key_pos)
    return (q_seq[:, None] == key_seq[None, :]) & (key_pos[None, :] <= q_pos[:, None])


def packed_key_layout(q_lens, context_lens):
    """Sequence id and position of every packed query row and of every key in the
    [cached keys of all requests | this step's new keys] layout."""
    key_seq, key_pos = [], []
    for r, c in enumerate(context_lens):
        key_seq += [r] * int(c)
        key_pos += list(range(int(c)))
    q_seq, q_pos = [], []
    for r, ql in enumerate(q_lens):
        for j in range(int(ql)):
            q_seq.append(r)
            q_pos.append(int(context_lens[r]) + j)
    return q_seq, q_pos, key_seq + q_seq, key_pos + q_pos


def attention_dense_mask(q, k_prior, v_prior, k_new, v_new, cu_seqlens_q, context_lens,
                         n_q_heads: int, n_kv_heads: int, head_dim: int, softmax_scale=None):
    """Brute-force packed attention with an explicit additive block-diagonal causal mask.

    Keys are laid out as [every request's cached keys | all new keys of this step]; each
    query row scores against all of them and masked entries get -inf before the
    softmax.  Small steps only: it is O(T * (sum ctx + T)).
    """
    d = head_dim
    group = n_q_heads // n_kv_heads
    scale = (1.0 / np.sqrt(float(d))) if softmax_scale is None else float(softmax_scale)
    q_lens = [int(cu_seqlens_q[r + 1] - cu_seqlens_q[r]) for r in range(len(context_lens))]
    q_seq, q_pos, key_seq, key_pos = packed_key_layout(q_lens, context_lens)
    allowed = block_diagonal_causal_mask(q_seq, q_pos, key_seq, key_pos)
    add_mask = np.where(allowed, 0.0, -np.inf)
    parts_k = [kp for kp in k_prior if kp is not None and kp.shape[0] > 0]
    parts_v = [vp for vp in v_prior if vp is not None and vp.shape[0] > 0]
    Kall = bf16_to_f64(np.concatenate(parts_k + [k_new], axis=0)).reshape(-1, n_kv_heads, d)
    Vall = bf16_to_f64(np.concatenate(parts_v + [v_new], axis=0)).reshape(-1, n_kv_heads, d)
    Q = bf16_to_f64(q).reshape(-1, n_q_heads, d)
    out = np.empty((Q.shape[0], n_q_heads, d), dtype=np.float64)
    for h in range(n_q_heads):
        kvh = h // group
        s = (Q[:, h, :] @ Kall[:, kvh, :].T) * scale + add_mask
        out[:, h, :] = softmax_weights(s) @ Vall[:, kvh, :]
    return out


# ----------------------------------------------------------------- full-step helpers

def request_histories(inp, requests=None):
    """Contiguous K and V history of every request (or of the listed ones; None for the
    others): cached tokens then this step's rows.

    `inp` is a StepInputs from the seeded generator.
    """
    ks, vs = [], []
    cu = inp.cu_seqlens_q
    for r in range(len(inp.context_lens)):
        s, e = int(cu[r]), int(cu[r + 1])
        kp, vp = inp.k_prior[r], inp.v_prior[r]
        if kp is None or (requests is not None and r not in requests):
            ks.append(None)
            vs.append(None)
            continue
        ks.append(np.concatenate([kp, inp.k_new[s:e]], axis=0))
        vs.append(np.concatenate([vp, inp.v_new[s:e]], axis=0))
    return ks, vs


def step_reference(inp, rows=None, softmax_scale=None):
    """Attention output of one whole step (or of the listed rows), fp64 [T, n_q, d]."""
    spec = inp.spec
    needed = None
    if rows is not None:   # only the requests that own a listed row
        cu = np.asarray(inp.cu_seqlens_q)
        needed = set(int(r) for r in np.searchsorted(cu, np.asarray(list(rows), dtype=np.int64), side="right") - 1)
    ks, vs = request_histories(inp, needed)
    return attention_reference(inp.q, ks, vs, inp.cu_seqlens_q, inp.context_lens,
                               spec.n_q_heads, spec.n_kv_heads, spec.head_dim,
                               softmax_scale=softmax_scale, rows=rows)
