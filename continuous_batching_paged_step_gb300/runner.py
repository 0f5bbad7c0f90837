"""Set up one packed step on the GPU and run it through the C ABI.

`PagedStep` owns a KV pool, places every request's blocks at the physical ids the step's
block tables name (kv_block_claim), writes each request's already-cached tokens into the
pool with kv_append (as an earlier prefill would have), and keeps the step's packed
tensors resident.  `run()` is one pass of the hot path: kv_append of this step's new
K/V, then paged_attention_step.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import kvpaged as kp
from .workloads import StepInputs


def _dev_bf16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def _dev_i32(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


class PagedStep:
    def __init__(self, inp: StepInputs, device="cuda", pool_fill_bits: int | None = None,
                 decode_ctas: int | None = None, fill_prior: bool = True, poison_workspace: bool = False,
                 mixed: bool = False):
        spec = inp.spec
        self.inp = inp
        self.device = device
        self.pool = kp.KVPool(spec.num_blocks, device=device)
        if pool_fill_bits is not None:
            fill = int(np.array([pool_fill_bits], dtype=np.uint16).view(np.int16)[0])
            self.pool.k_cache.view(torch.int16).fill_(fill)
            self.pool.v_cache.view(torch.int16).fill_(fill)
        if decode_ctas is not None:
            kp.kv_pool_set_decode_ctas(self.pool.handle, decode_ctas)
        if mixed:
            kp.kv_pool_set_step_kernel(self.pool.handle, True)
        kp.kv_block_claim(self.pool.handle, inp.block_order)
        self.block_tables = _dev_i32(inp.block_tables, device)
        self.cu_seqlens_q = _dev_i32(inp.cu_seqlens_q, device)
        self.context_lens = _dev_i32(inp.context_lens, device)
        self.q = _dev_bf16(inp.q, device)
        self.k_new = _dev_bf16(inp.k_new, device)
        self.v_new = _dev_bf16(inp.v_new, device)
        self.out = torch.zeros_like(self.q)
        self.max_q_len = int(max(spec.q_lens)) if spec.q_lens else 0
        self.max_context_len = int(max(spec.ctx_lens)) if spec.ctx_lens else 0
        self.softmax_scale = 1.0 / math.sqrt(spec.head_dim)
        ws = kp.paged_attention_workspace_size(self.pool.handle, spec.num_reqs, spec.num_tokens,
                                               self.max_context_len)
        self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=device)
        if poison_workspace:
            self.workspace.fill_(0x5A)        # stale-looking bytes: nothing may read scratch it did not write
        if fill_prior:
            self.write_prior()

    def write_prior(self):
        """Write every request's cached tokens (positions 0..ctx-1) into the pool."""
        inp = self.inp
        ctx = inp.context_lens.astype(np.int64)
        if ctx.sum() == 0:
            return
        parts_k = [kp_ for kp_ in inp.k_prior if kp_ is not None and kp_.shape[0] > 0]
        parts_v = [vp for vp in inp.v_prior if vp is not None and vp.shape[0] > 0]
        if sum(p.shape[0] for p in parts_k) != ctx.sum():
            raise ValueError("prior K/V of every request is needed to fill the pool")
        cu = np.zeros(len(ctx) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(ctx)
        k = _dev_bf16(np.concatenate(parts_k), self.device)
        v = _dev_bf16(np.concatenate(parts_v), self.device)
        kp.kv_append(self.pool.handle, k, v, _dev_i32(cu, self.device),
                     torch.zeros(len(ctx), dtype=torch.int32, device=self.device), self.block_tables)
        del k, v

    def append(self, stream=None):
        kp.kv_append(self.pool.handle, self.k_new, self.v_new, self.cu_seqlens_q, self.context_lens,
                     self.block_tables, stream=stream)

    def attend(self, stream=None):
        kp.paged_attention_step(self.pool.handle, self.q, self.out, self.cu_seqlens_q, self.context_lens,
                                self.block_tables, self.max_q_len, self.max_context_len, self.softmax_scale,
                                self.workspace, stream=stream)

    def run(self, stream=None):
        self.append(stream)
        self.attend(stream)

    def error(self, stream=None):
        return kp.kv_pool_get_error(self.pool.handle, stream)

    def out_f32(self) -> np.ndarray:
        spec = self.inp.spec
        return self.out.float().cpu().numpy().reshape(spec.num_tokens, spec.n_q_heads, spec.head_dim)

    def close(self):
        self.pool.close()
