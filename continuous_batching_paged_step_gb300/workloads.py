"""Seeded synthetic inputs for one packed continuous-batching step.

This module is the only code shared by the CUDA path (tests, bench) and the
CPU oracle.  It draws numbers and lays out integer metadata; it holds none of
the method's arithmetic (no slot mapping, no masking, no attention).

Shapes follow the mixed-batch example of page "11.2 连续批处理与 PagedAttention"
(section 11.2.2, Figure 11-3): Q rows are [T, n_q*128] and new K/V rows are
[T, n_kv*128] with head h occupying columns [h*128, (h+1)*128).  bf16 values
are carried as uint16 bit patterns, drawn as float32 N(0, 1) and rounded to
nearest-even.

Every array of request r is drawn from its own stream, seeded by
(step seed, r, stream kind), so any subset of requests can be regenerated
alone and large steps can be generated on several threads.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16
N_Q_HEADS = 32
N_KV_HEADS = 8
HEAD_DIM = 128

_KIND_Q, _KIND_KNEW, _KIND_VNEW, _KIND_KPRIOR, _KIND_VPRIOR = range(5)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(seed: int, r: int, kind: int, shape) -> np.ndarray:
    rng = np.random.default_rng([seed, r, kind])
    n = int(np.prod(shape))
    return f32_to_bf16_bits(rng.standard_normal(n, dtype=np.float32)).reshape(shape)


@dataclass
class StepSpec:
    """One packed step: request r brings q_lens[r] new rows after ctx_lens[r] cached tokens."""
    name: str
    q_lens: list
    ctx_lens: list
    num_blocks: int
    seed: int
    n_q_heads: int = N_Q_HEADS
    n_kv_heads: int = N_KV_HEADS
    head_dim: int = HEAD_DIM
    block_size: int = BLOCK_SIZE
    extra: dict = field(default_factory=dict)

    @property
    def num_reqs(self) -> int:
        return len(self.q_lens)

    @property
    def num_tokens(self) -> int:
        return int(sum(self.q_lens))

    def blocks_needed(self, r: int) -> int:
        return -(-(self.ctx_lens[r] + self.q_lens[r]) // self.block_size)

    @property
    def max_blocks_per_seq(self) -> int:
        return max(1, max(self.blocks_needed(r) for r in range(self.num_reqs)))


@dataclass
class StepInputs:
    spec: StepSpec
    q: np.ndarray              # uint16 [T, n_q*d]
    k_new: np.ndarray          # uint16 [T, n_kv*d]
    v_new: np.ndarray          # uint16 [T, n_kv*d]
    k_prior: list              # per request uint16 [ctx_r, n_kv*d]
    v_prior: list
    cu_seqlens_q: np.ndarray   # int32 [R+1]
    context_lens: np.ndarray   # int32 [R]
    block_tables: np.ndarray   # int32 [R, max_blocks]; unused entries are -1
    block_order: np.ndarray    # int32: physical ids in the order they were handed out


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def make_inputs(spec: StepSpec, with_prior: bool = True, requests=None) -> StepInputs:
    """Draw every array of the step.  `requests` restricts the per-request prior K/V
    (the packed Q/K/V rows are always complete); other prior entries are None."""
    R, T = spec.num_reqs, spec.num_tokens
    hq, hk, d = spec.n_q_heads, spec.n_kv_heads, spec.head_dim
    cu = np.zeros(R + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(spec.q_lens, dtype=np.int64))
    ctx = np.asarray(spec.ctx_lens, dtype=np.int32)

    perm = np.random.default_rng([spec.seed, 0x7AB1E]).permutation(spec.num_blocks).astype(np.int32)
    need = [spec.blocks_needed(r) for r in range(R)]
    if sum(need) > spec.num_blocks:
        raise ValueError(f"{spec.name}: {sum(need)} blocks needed, pool has {spec.num_blocks}")
    tables = np.full((R, spec.max_blocks_per_seq), -1, dtype=np.int32)
    off = 0
    for r in range(R):
        tables[r, :need[r]] = perm[off:off + need[r]]
        off += need[r]

    def rows(r):
        ql = spec.q_lens[r]
        return (_normal_bf16(spec.seed, r, _KIND_Q, (ql, hq * d)),
                _normal_bf16(spec.seed, r, _KIND_KNEW, (ql, hk * d)),
                _normal_bf16(spec.seed, r, _KIND_VNEW, (ql, hk * d)))

    want = set(range(R)) if requests is None else set(requests)

    def prior(r):
        if not with_prior or r not in want:
            return None, None
        c = spec.ctx_lens[r]
        return (_normal_bf16(spec.seed, r, _KIND_KPRIOR, (c, hk * d)),
                _normal_bf16(spec.seed, r, _KIND_VPRIOR, (c, hk * d)))

    with ThreadPoolExecutor(_threads()) as ex:
        new_rows = list(ex.map(rows, range(R)))
        priors = list(ex.map(prior, range(R)))

    def cat(i, width):
        parts = [nr[i] for nr in new_rows if nr[i].shape[0] > 0]
        return np.concatenate(parts, axis=0) if parts else np.zeros((0, width), np.uint16)

    return StepInputs(spec=spec, q=cat(0, hq * d), k_new=cat(1, hk * d), v_new=cat(2, hk * d),
                      k_prior=[p[0] for p in priors], v_prior=[p[1] for p in priors],
                      cu_seqlens_q=cu, context_lens=ctx, block_tables=tables,
                      block_order=perm[:off].copy())


# --------------------------------------------------------------------------------------
# The step shapes.  Sizes follow the workloads described for the method: the 3-request
# mixed step of page "11.2 连续批处理与 PagedAttention" (section 11.2.2), decode rows over
# long cached histories, and chunked prefill under an 8192-token budget (section 11.2.5).
# --------------------------------------------------------------------------------------

def tiny_p5_step(seed: int = 0xC0FFEE + 1) -> StepSpec:
    """R1 prefills 5 tokens with nothing cached; R2 and R3 decode one token after 7 and 3
    cached tokens; pool of 64 blocks."""
    return StepSpec("tiny-3req", q_lens=[5, 1, 1], ctx_lens=[0, 7, 3], num_blocks=64, seed=seed)


def mixed_step(seed: int = 0xC0FFEE + 2) -> StepSpec:
    """64 decode rows with context ~ U[128, 4096] plus two 512-token prefill chunks with
    0 and 1024 tokens cached; pool of 32768 blocks."""
    rng = np.random.default_rng([seed, 1])
    dec_ctx = rng.integers(128, 4096, size=64, endpoint=True).tolist()
    return StepSpec("mixed-64dec-2x512", q_lens=[1] * 64 + [512, 512],
                    ctx_lens=dec_ctx + [0, 1024], num_blocks=32768, seed=seed)


def decode_heavy_step(seed: int = 0xC0FFEE + 3, num_blocks: int = 32768) -> StepSpec:
    """256 decode rows, context lognormal with median 1024 and sigma 0.8, clipped to [16, 8192]."""
    rng = np.random.default_rng([seed, 1])
    ctx = np.clip(np.round(np.exp(math.log(1024.0) + 0.8 * rng.standard_normal(256))), 16, 8192)
    return StepSpec("decode-256-lognormal", q_lens=[1] * 256, ctx_lens=ctx.astype(int).tolist(),
                    num_blocks=num_blocks, seed=seed)


def chunked_prefill_step(seed: int = 0xC0FFEE + 4, num_blocks: int = 32768) -> StepSpec:
    """Four 2048-token prefill chunks with 0/2048/4096/6144 cached, plus 32 decode rows
    with context ~ U[512, 8192] (8224 packed rows)."""
    rng = np.random.default_rng([seed, 1])
    dec_ctx = rng.integers(512, 8192, size=32, endpoint=True).tolist()
    return StepSpec("chunked-4x2048-32dec", q_lens=[2048] * 4 + [1] * 32,
                    ctx_lens=[0, 2048, 4096, 6144] + dec_ctx, num_blocks=num_blocks, seed=seed)


def small_mixed_step(seed: int = 0xC0FFEE + 9, n_decode: int = 12, chunks=((200, 37), (130, 0)),
                     ctx_range=(1, 700), num_blocks: int = 1024) -> StepSpec:
    """A small mixed step for the oracle's element-by-element comparison: several decode
    rows, prefill chunks spanning more than one 128-row tile with a ragged tail, block
    boundaries crossed at odd offsets."""
    rng = np.random.default_rng([seed, 1])
    dec_ctx = rng.integers(ctx_range[0], ctx_range[1], size=n_decode, endpoint=True).tolist()
    q_lens = [1] * n_decode + [c[0] for c in chunks]
    ctx = dec_ctx + [c[1] for c in chunks]
    return StepSpec("small-mixed", q_lens=q_lens, ctx_lens=ctx, num_blocks=num_blocks, seed=seed)


CONFIGS = {
    "tiny": tiny_p5_step,
    "mixed": mixed_step,
    "decode": decode_heavy_step,
    "chunked": chunked_prefill_step,
}


# --------------------------------------------------------------------------------------
# Trace replay: a stream of requests arriving over steps.  Lengths follow the shapes named
# for the method's workloads (page "11.2 连续批处理与 PagedAttention", sections 11.2.2-11.2.5):
# a shared system prompt, skewed prompt and output lengths.  Values the pages leave open
# (arrival rate, lognormal sigmas) are fixed here and recorded with the design.
# --------------------------------------------------------------------------------------

@dataclass
class TraceSpec:
    name: str = "trace-512req"
    n_requests: int = 512
    arrivals_per_step: float = 4.0        # Poisson rate on the step clock
    shared_prefix: int = 1024             # tokens of the shared system prompt (full blocks)
    prompt_median: float = 256.0
    prompt_sigma: float = 1.0
    prompt_cap: int = 4096
    output_median: float = 100.0
    output_sigma: float = 1.0
    output_range: tuple = (10, 2000)
    budget: int = 8192                    # tokens per step, decode rows first
    max_num_seqs: int = 0                 # 0: no limit on running requests
    pool_blocks: int = 655360             # 40 GiB of K+V for one layer
    seed: int = 0xC0FFEE + 5


@dataclass
class TraceRequest:
    rid: int
    arrival: int          # step at which the request becomes visible to the scheduler
    prompt_len: int       # own prompt tokens, after the shared prefix
    output_len: int       # tokens the request generates (the first comes with its last prefill chunk)


def make_trace(ts: TraceSpec) -> list:
    rng = np.random.default_rng([ts.seed, 0x7EACE])
    reqs, step = [], 0
    while len(reqs) < ts.n_requests:
        for _ in range(int(rng.poisson(ts.arrivals_per_step))):
            if len(reqs) == ts.n_requests:
                break
            p = int(np.clip(np.round(np.exp(math.log(ts.prompt_median) + ts.prompt_sigma * rng.standard_normal())),
                            1, ts.prompt_cap))
            o = int(np.clip(np.round(np.exp(math.log(ts.output_median) + ts.output_sigma * rng.standard_normal())),
                            ts.output_range[0], ts.output_range[1]))
            reqs.append(TraceRequest(len(reqs), step, p, o))
        step += 1
    return reqs


_TRACE_Q, _TRACE_K, _TRACE_V = 11, 12, 13


def trace_rows(seed: int, rid: int, start: int, n: int, n_q: int = N_Q_HEADS * HEAD_DIM,
               n_kv: int = N_KV_HEADS * HEAD_DIM):
    """Q, K and V rows (bf16 bits) of the n tokens a request feeds from position `start`.
    rid = -1 is the shared system prompt.  Each (request, start) chunk has its own stream,
    so any chunk can be regenerated alone."""
    return (_normal_bf16(seed, rid + 1, _TRACE_Q * 100003 + start, (n, n_q)),
            _normal_bf16(seed, rid + 1, _TRACE_K * 100003 + start, (n, n_kv)),
            _normal_bf16(seed, rid + 1, _TRACE_V * 100003 + start, (n, n_kv)))


# --------------------------------------------------------------------------------------
# Shaped inputs for sensitive parity checks.  With N(0, 1) queries and keys the scores
# are ~N(0, 1), attention is close to uniform over a long history, and one 16-key block
# more or less moves a row's output by less than the comparison tolerance.  These
# shapers move input values only (no attention arithmetic): they add a per-(request,
# KV group) direction d to the query rows and place keys along it, so that chosen keys
# dominate every row's weights ("needles") or so that scores climb along the history
# (the running maximum keeps moving until the last keys).
# --------------------------------------------------------------------------------------

def long_context_step(seed: int = 0xC0FFEE + 21) -> StepSpec:
    """Decode rows over contexts from 0 to 8192 (block-boundary values included) and
    prefill chunks after long cached prefixes: 2048 rows after 6144, 300 after 4000, 130
    after nothing and 33 after 127 (a chunk that starts one key before a 128-key tile)."""
    rng = np.random.default_rng([seed, 1])
    dec = [8192, 8191, 8177, 8176, 6000, 4096, 4095, 3333, 2048, 1024, 1023, 767, 512, 511, 300, 257, 256,
           255, 100, 31, 16, 15, 1, 0]
    dec += rng.integers(1, 8192, size=8, endpoint=True).tolist()
    chunks = [(2048, 6144), (300, 4000), (130, 0), (33, 127)]
    q_lens = [1] * len(dec) + [c[0] for c in chunks]
    ctx = dec + [c[1] for c in chunks]
    # interleave the chunks among the decode rows so request order is mixed
    order = np.random.default_rng([seed, 2]).permutation(len(q_lens)).tolist()
    q_lens = [q_lens[i] for i in order]
    ctx = [ctx[i] for i in order]
    need = sum(-(-(c + q) // BLOCK_SIZE) for c, q in zip(ctx, q_lens))
    return StepSpec("long-context", q_lens=q_lens, ctx_lens=ctx, num_blocks=need + 97, seed=seed)


def _as_f32(bits):
    return bf16_bits_to_f32(bits).copy()


def _key_row(inp: StepInputs, r: int, t: int, which: str):
    """(array, row index) holding position t of request r's K (which='k') or V history."""
    ctx = int(inp.context_lens[r])
    if t < ctx:
        return (inp.k_prior if which == "k" else inp.v_prior)[r], t
    return (inp.k_new if which == "k" else inp.v_new), int(inp.cu_seqlens_q[r]) + t - ctx


def _copy_inputs(inp: StepInputs) -> StepInputs:
    return StepInputs(spec=inp.spec, q=inp.q.copy(), k_new=inp.k_new.copy(), v_new=inp.v_new.copy(),
                      k_prior=[None if a is None else a.copy() for a in inp.k_prior],
                      v_prior=[None if a is None else a.copy() for a in inp.v_prior],
                      cu_seqlens_q=inp.cu_seqlens_q, context_lens=inp.context_lens,
                      block_tables=inp.block_tables, block_order=inp.block_order)


def _directions(spec: StepSpec, seed: int):
    """A unit-variance direction per (request, KV group): float32 [R, n_kv, d]."""
    rng = np.random.default_rng([seed, 0xD1])
    return rng.standard_normal((spec.num_reqs, spec.n_kv_heads, spec.head_dim)).astype(np.float32)


def _add_to_queries(out: StepInputs, d, beta: float):
    """Query rows of request r, every head of KV group g: q += beta * d[r, g]."""
    spec = out.spec
    g = spec.n_q_heads // spec.n_kv_heads
    q = _as_f32(out.q).reshape(-1, spec.n_kv_heads, g, spec.head_dim)
    cu = out.cu_seqlens_q
    for r in range(spec.num_reqs):
        s, e = int(cu[r]), int(cu[r + 1])
        if e > s:
            q[s:e] += beta * d[r][None, :, None, :]
    out.q = f32_to_bf16_bits(q.reshape(out.q.shape))


def needle_positions(spec: StepSpec, every_block_max: int = 48, spread: int = 16):
    """Key positions planted as needles, per request.  A history of at most
    `every_block_max` blocks gets one needle in every block (offsets inside the block
    cycle through 0, 15, 7, 8, 3, 12, ...); a longer one gets `spread` needles in blocks
    spread evenly from its first to its last block, offsets alternating 0 and 15."""
    offs = [0, 15, 7, 8, 3, 12, 1, 14, 5, 10]
    out = []
    for r in range(spec.num_reqs):
        n = spec.ctx_lens[r] + spec.q_lens[r]
        if spec.q_lens[r] == 0 or n == 0:
            out.append([])
            continue
        nb = -(-n // spec.block_size)
        if nb <= every_block_max:
            blocks = list(range(nb))
        else:
            blocks = sorted(set(int(round(k * (nb - 1) / (spread - 1))) for k in range(spread)))
        pos = []
        for i, b in enumerate(blocks):
            o = offs[i % len(offs)] if nb <= every_block_max else (0 if i % 2 == 0 else 15)
            pos.append(min(b * spec.block_size + o, n - 1))
        out.append(sorted(set(pos)))
    return out


def plant_needles(inp: StepInputs, alpha: float = 0.5, beta: float = 4.0, v_scale: float = 0.5,
                  seed: int = 0xBEEF, positions=None):
    """Needle inputs: query rows of request r get beta * d[r, g] added on every head of
    KV group g; the key at each needle position becomes alpha * d[r, g] (so its score,
    about alpha * beta * d . d / sqrt(d), is far above the other keys' for every row that
    sees it) and its value is scaled by v_scale (keeps outputs near the values' scale).
    Returns (inputs, positions)."""
    spec = inp.spec
    out = _copy_inputs(inp)
    d = _directions(spec, seed)
    _add_to_queries(out, d, beta)
    pos = needle_positions(spec) if positions is None else positions
    for r, ps in enumerate(pos):
        for t in ps:
            ka, ki = _key_row(out, r, t, "k")
            ka[ki] = f32_to_bf16_bits((alpha * d[r]).reshape(-1))
            va, vi = _key_row(out, r, t, "v")
            va[vi] = f32_to_bf16_bits(_as_f32(va[vi]) * np.float32(v_scale))
    return out, pos


def plant_late_peak(inp: StepInputs, gamma_max: float = 5.0, beta: float = 1.0, v_scale: float = 0.5,
                    seed: int = 0xFEED):
    """Late-peak inputs: query rows of request r get beta * d[r, g] added; the key at
    position t of a history of n keys gets gamma_max * t / (n - 1) * d[r, g] added, so
    scores climb by tens of units along the history and the running maximum keeps
    moving until the last keys.  Values are scaled by v_scale."""
    spec = inp.spec
    out = _copy_inputs(inp)
    d = _directions(spec, seed)
    _add_to_queries(out, d, beta)
    kn = _as_f32(out.k_new).reshape(-1, spec.n_kv_heads, spec.head_dim)
    cu = out.cu_seqlens_q
    for r in range(spec.num_reqs):
        c, ql = spec.ctx_lens[r], spec.q_lens[r]
        n = c + ql
        if ql == 0 or n < 2:
            continue
        ramp = (gamma_max * np.arange(n, dtype=np.float32) / np.float32(n - 1))[:, None, None] * d[r][None]
        if c > 0:
            kp = _as_f32(out.k_prior[r]).reshape(c, spec.n_kv_heads, spec.head_dim) + ramp[:c]
            out.k_prior[r] = f32_to_bf16_bits(kp.reshape(c, -1))
            out.v_prior[r] = f32_to_bf16_bits(_as_f32(out.v_prior[r]) * np.float32(v_scale))
        s = int(cu[r])
        kn[s:s + ql] += ramp[c:]
    out.k_new = f32_to_bf16_bits(kn.reshape(out.k_new.shape))
    out.v_new = f32_to_bf16_bits(_as_f32(out.v_new) * np.float32(v_scale))
    return out
