"""Thin Python binding of libkvpaged.so (the C ABI in include/kvpaged.h).

Argument marshalling only: every step of the path runs in the library's CUDA kernels.
PyTorch supplies device memory and streams.  Importing this module fails loudly when
the library has not been built; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libkvpaged.so")

KVP_OK = 0
STATUS_NAMES = {0: "KVP_OK", -1: "KVP_E_INVALID_ARG", -2: "KVP_E_NO_BLOCKS", -3: "KVP_E_BAD_BLOCK",
                -4: "KVP_E_SHARED_WRITE", -5: "KVP_E_BAD_META", -6: "KVP_E_CUDA", -7: "KVP_E_REFCOUNT",
                -8: "KVP_E_WORKSPACE", -9: "KVP_E_TIMEOUT"}
ERRBIT_BAD_BLOCK, ERRBIT_SHARED_WRITE, ERRBIT_BAD_META, ERRBIT_TIMEOUT = 0x1, 0x2, 0x4, 0x8
DTYPE_BF16 = 1
BLOCK_SIZE, N_KV_HEADS, N_Q_HEADS, HEAD_DIM = 16, 8, 32, 128

# every symbol include/kvpaged.h declares, with (restype, argtypes)
_P, _I, _SZ, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
_I32P = ctypes.POINTER(ctypes.c_int32)
SIGNATURES = {
    "kv_pool_create": (_I, [_I, _I, _I, _I, _I, _P, _P, ctypes.POINTER(_P)]),
    "kv_pool_destroy": (_I, [_P]),
    "kv_block_alloc": (_I, [_P, _I, _I32P]),
    "kv_block_claim": (_I, [_P, _I, _I32P]),
    "kv_block_ref": (_I, [_P, _I, _I32P]),
    "kv_block_free": (_I, [_P, _I, _I32P]),
    "kv_pool_num_free": (_I, [_P]),
    "kv_block_refcount": (_I, [_P, ctypes.c_int32]),
    "kv_append": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "paged_attention_workspace_size": (_SZ, [_P, _I, _I, _I, _I]),
    "paged_attention_step": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _SZ, _P]),
    "kv_pool_set_decode_ctas": (_I, [_P, _I]),
    "kv_pool_set_step_kernel": (_I, [_P, _I]),
    "kv_pool_set_nvtx": (_I, [_P, _I]),
    "kv_pool_get_error": (_I, [_P, _P, ctypes.POINTER(ctypes.c_uint32)]),
    "kvp_status_string": (ctypes.c_char_p, [_I]),
    "kv_pool_enable_timing": (_I, [_P, _I]),
    "kv_pool_read_timing": (_I, [_P, ctypes.POINTER(_I), ctypes.POINTER(_F)]),
    "kv_pool_launch_count": (ctypes.c_longlong, [_P]),
    "paged_attention_step_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "paged_attention_noalloc_capacity": (_SZ, []),
    "kvp_selftest_bounded_wait": (_I, [ctypes.c_longlong, _P]),
    "kv_block_cow": (_I, [_P, _I, _I32P, _I32P, _P]),
    "kv_blocks_swap_out": (_I, [_P, _I, _I32P, _P, _P, _P]),
    "kv_blocks_swap_in": (_I, [_P, _I, _P, _P, _I32P, _P]),
}
KERNEL_NAMES = ("kv_append", "step_prep", "prefill_tcgen05", "decode_splitkv", "block_move", "splitkv_combine",
                "mixed_step")
BLOCK_BYTES = N_KV_HEADS * BLOCK_SIZE * HEAD_DIM * 2   # one block of K (or of V): 32 KiB


class KVPError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def _check(status: int, what: str):
    if status != KVP_OK:
        raise KVPError(status, what)


def _ids(ids):
    a = np.ascontiguousarray(np.asarray(ids, dtype=np.int32).reshape(-1))
    return a, a.ctypes.data_as(_I32P)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t, dtype, what):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{what} must be a contiguous CUDA tensor of {dtype}")


# ------------------------------------------------------------------------ pool

def kv_pool_create(k_cache, v_cache, num_blocks: int | None = None) -> int:
    """Wrap caller-owned pools bf16 [num_blocks, 8, 16, 128]; returns the pool handle.
    k_cache/v_cache may be raw device addresses (int) when num_blocks is given."""
    if isinstance(k_cache, int):
        nb = int(num_blocks)
    else:
        import torch
        _need(k_cache, torch.bfloat16, "k_cache")
        _need(v_cache, torch.bfloat16, "v_cache")
        if tuple(k_cache.shape[1:]) != (N_KV_HEADS, BLOCK_SIZE, HEAD_DIM) or k_cache.shape != v_cache.shape:
            raise ValueError("pools must be [num_blocks, 8, 16, 128]")
        nb = k_cache.shape[0]
    h = _P()
    _check(lib.kv_pool_create(nb, BLOCK_SIZE, N_KV_HEADS, HEAD_DIM, DTYPE_BF16, _ptr(k_cache), _ptr(v_cache),
                              ctypes.byref(h)), "kv_pool_create")
    return h.value


def kv_pool_destroy(pool: int):
    _check(lib.kv_pool_destroy(pool), "kv_pool_destroy")


def kv_block_alloc(pool: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _check(lib.kv_block_alloc(pool, n, out.ctypes.data_as(_I32P)), "kv_block_alloc")
    return out


def kv_block_claim(pool: int, ids):
    a, p = _ids(ids)
    _check(lib.kv_block_claim(pool, a.size, p), "kv_block_claim")


def kv_block_ref(pool: int, ids):
    a, p = _ids(ids)
    _check(lib.kv_block_ref(pool, a.size, p), "kv_block_ref")


def kv_block_free(pool: int, ids):
    a, p = _ids(ids)
    _check(lib.kv_block_free(pool, a.size, p), "kv_block_free")


def _stream_or_null(stream):
    """The stream handle, or None (the legacy default stream) when torch has no CUDA."""
    if stream is not None:
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    import torch
    return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None


def kv_block_cow(pool: int, src_ids, stream=None) -> np.ndarray:
    """Copy-on-write: for each listed block, the block itself if its refcount is 1, else a
    new block holding a copy of it (the source loses one reference)."""
    a, p = _ids(src_ids)
    out = np.empty(a.size, dtype=np.int32)
    _check(lib.kv_block_cow(pool, a.size, p, out.ctypes.data_as(_I32P), _stream_or_null(stream)), "kv_block_cow")
    return out


def _pinned(t, n: int, what: str):
    import torch
    if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_pinned() or not t.is_contiguous():
        raise ValueError(f"{what} must be a contiguous pinned host tensor")
    if t.numel() * t.element_size() < n * BLOCK_BYTES:
        raise ValueError(f"{what} holds fewer than {n} blocks")


def kv_blocks_swap_out(pool: int, ids, host_k, host_v, stream=None):
    """Copy the listed blocks' K and V to pinned host tensors (block i at byte i * 32 KiB)
    and release one reference of each."""
    a, p = _ids(ids)
    _pinned(host_k, a.size, "host_k")
    _pinned(host_v, a.size, "host_v")
    _check(lib.kv_blocks_swap_out(pool, a.size, p, _ptr(host_k), _ptr(host_v), _stream(stream)),
           "kv_blocks_swap_out")


def kv_blocks_swap_in(pool: int, host_k, host_v, n: int, stream=None) -> np.ndarray:
    """Allocate n blocks and copy block i of the pinned host tensors into them; returns
    the new block ids."""
    _pinned(host_k, n, "host_k")
    _pinned(host_v, n, "host_v")
    out = np.empty(n, dtype=np.int32)
    _check(lib.kv_blocks_swap_in(pool, n, _ptr(host_k), _ptr(host_v), out.ctypes.data_as(_I32P), _stream(stream)),
           "kv_blocks_swap_in")
    return out


def kv_pool_num_free(pool: int) -> int:
    return lib.kv_pool_num_free(pool)


def kv_block_refcount(pool: int, block_id: int) -> int:
    return lib.kv_block_refcount(pool, block_id)


def kv_pool_set_decode_ctas(pool: int, ctas: int):
    """Number of CTAs the decode blocks are shared out among (0 = one per SM)."""
    _check(lib.kv_pool_set_decode_ctas(pool, ctas), "kv_pool_set_decode_ctas")


def kv_pool_set_nvtx(pool: int, on: bool):
    """NVTX ranges (domain "kvpaged") around this pool's calls and kernel launches."""
    _check(lib.kv_pool_set_nvtx(pool, 1 if on else 0), "kv_pool_set_nvtx")


def kv_pool_set_step_kernel(pool: int, mixed: bool):
    """Run the step's attention as the mixed step kernel (one grid, work tickets) instead
    of the decode kernel and the prefill kernel side by side."""
    _check(lib.kv_pool_set_step_kernel(pool, 1 if mixed else 0), "kv_pool_set_step_kernel")


def kv_pool_get_error(pool: int, stream=None):
    """Synchronise the stream, read and clear the device error word: (status, bits)."""
    bits = ctypes.c_uint32(0)
    st = lib.kv_pool_get_error(pool, _stream(stream), ctypes.byref(bits))
    return st, bits.value


def kv_pool_enable_timing(pool: int, max_launches: int):
    _check(lib.kv_pool_enable_timing(pool, max_launches), "kv_pool_enable_timing")


def kv_pool_read_timing(pool: int):
    """{kernel name: (timed launches, summed ms)} since the last read."""
    counts = (_I * len(KERNEL_NAMES))()
    ms = (_F * len(KERNEL_NAMES))()
    _check(lib.kv_pool_read_timing(pool, counts, ms), "kv_pool_read_timing")
    return {n: (counts[i], ms[i]) for i, n in enumerate(KERNEL_NAMES)}


def kv_pool_launch_count(pool: int) -> int:
    return lib.kv_pool_launch_count(pool)


def kvp_selftest_bounded_wait(limit_ns: int, stream=None) -> int:
    """Make one bounded device wait run out on purpose; returns the status (KVP_E_TIMEOUT
    when the wait gave up as it should)."""
    return lib.kvp_selftest_bounded_wait(int(limit_ns), _stream(stream))


# ------------------------------------------------------------------ the step

def kv_append(pool: int, k_new, v_new, cu_seqlens_q, context_lens, block_tables, stream=None):
    """Append this step's K/V rows (bf16 [T, 1024]) into the pool."""
    import torch
    T = k_new.shape[0]
    if T:
        _need(k_new, torch.bfloat16, "k_new")
        _need(v_new, torch.bfloat16, "v_new")
        for t, n in ((cu_seqlens_q, "cu_seqlens_q"), (context_lens, "context_lens"), (block_tables, "block_tables")):
            _need(t, torch.int32, n)
    R = context_lens.shape[0]
    _check(lib.kv_append(pool, _ptr(k_new), _ptr(v_new), _ptr(cu_seqlens_q), _ptr(context_lens),
                         _ptr(block_tables), block_tables.shape[1], R, T, _stream(stream)), "kv_append")


def paged_attention_workspace_size(pool: int, num_reqs: int, num_tokens: int, max_context_len: int) -> int:
    return lib.paged_attention_workspace_size(pool, num_reqs, num_tokens, N_Q_HEADS, max_context_len)


def paged_attention_step(pool: int, q, out, cu_seqlens_q, context_lens, block_tables, max_q_len: int,
                         max_context_len: int, softmax_scale: float, workspace, stream=None):
    """Varlen paged attention of the packed rows q (bf16 [T, 4096]) into out (same shape)."""
    import torch
    T = q.shape[0]
    if T:
        _need(q, torch.bfloat16, "q")
        _need(out, torch.bfloat16, "out")
        _need(workspace, torch.uint8, "workspace")
        for t, n in ((cu_seqlens_q, "cu_seqlens_q"), (context_lens, "context_lens"), (block_tables, "block_tables")):
            _need(t, torch.int32, n)
    R = context_lens.shape[0]
    _check(lib.paged_attention_step(pool, _ptr(q), _ptr(out), _ptr(cu_seqlens_q), _ptr(context_lens),
                                    _ptr(block_tables), block_tables.shape[1], R, T, N_Q_HEADS, max_q_len,
                                    max_context_len, float(softmax_scale), _ptr(workspace),
                                    workspace.numel() if workspace is not None else 0, _stream(stream)),
           "paged_attention_step")


class KVPool:
    """Owns a pair of device pools and the library handle for them."""

    def __init__(self, num_blocks: int, device="cuda"):
        import torch
        shape = (num_blocks, N_KV_HEADS, BLOCK_SIZE, HEAD_DIM)
        self.k_cache = torch.empty(shape, dtype=torch.bfloat16, device=device)
        self.v_cache = torch.empty(shape, dtype=torch.bfloat16, device=device)
        self.num_blocks = num_blocks
        self.handle = kv_pool_create(self.k_cache, self.v_cache)

    def close(self):
        if self.handle:
            kv_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def paged_attention_step_noalloc(pool: int, q, out, cu_seqlens_q, context_lens, block_tables, max_q_len: int,
                                 max_context_len: int, softmax_scale: float, stream=None):
    """paged_attention_step without a caller workspace: the library's fixed scratch array
    is used instead, so the call allocates no device memory (see include/kvpaged.h)."""
    import torch
    T = q.shape[0]
    if T:
        _need(q, torch.bfloat16, "q")
        _need(out, torch.bfloat16, "out")
        for t, n in ((cu_seqlens_q, "cu_seqlens_q"), (context_lens, "context_lens"), (block_tables, "block_tables")):
            _need(t, torch.int32, n)
    R = context_lens.shape[0]
    _check(lib.paged_attention_step_noalloc(pool, _ptr(q), _ptr(out), _ptr(cu_seqlens_q), _ptr(context_lens),
                                            _ptr(block_tables), block_tables.shape[1], R, T, N_Q_HEADS, max_q_len,
                                            max_context_len, float(softmax_scale), _stream(stream)),
           "paged_attention_step_noalloc")


def paged_attention_noalloc_capacity() -> int:
    return lib.paged_attention_noalloc_capacity()
