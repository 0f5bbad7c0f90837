"""CPU checks of the C-ABI library: it builds, loads, exports every declared symbol, and
its host-side block allocator behaves as the block manager described for PagedAttention
(free list, refcounts, shared blocks, all-or-nothing errors).  No compute call is made."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kp():
    from continuous_batching_paged_step_gb300 import build
    build.build()
    from continuous_batching_paged_step_gb300 import kvpaged
    return kvpaged


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "kvpaged.h"), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*KVP_API\s+(?:[A-Za-z_][A-Za-z0-9_]*\s+)*?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*"
                       r"([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary_calls():
    names = _declared_functions()
    for want in ("kv_pool_create", "kv_pool_destroy", "kv_append", "paged_attention_step",
                 "paged_attention_workspace_size", "kv_block_alloc", "kv_block_ref", "kv_block_free",
                 "kv_pool_get_error"):
        assert want in names


def test_library_exports_every_declared_symbol(kp):
    lib = ctypes.CDLL(kp.LIB_PATH)
    names = _declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), n
        assert n in kp.SIGNATURES, f"binding lacks {n}"
    assert set(kp.SIGNATURES) == set(names)


def test_no_kernel_or_internal_symbol_is_exported(kp):
    out = os.popen(f"nm -D --defined-only {kp.LIB_PATH}").read()
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(_declared_functions())


FAKE_K, FAKE_V = 0x7F0000000000, 0x7F8000000000   # aligned addresses; create() touches no CUDA


def _pool(kp, nb=8):
    return kp.kv_pool_create(FAKE_K, FAKE_V, num_blocks=nb)


def test_create_validates_geometry(kp):
    h = ctypes.c_void_p()
    lib = kp.lib
    assert lib.kv_pool_create(8, 16, 8, 128, 1, FAKE_K, FAKE_V, ctypes.byref(h)) == 0
    lib.kv_pool_destroy(h)
    for args in ((8, 32, 8, 128, 1), (8, 16, 4, 128, 1), (8, 16, 8, 64, 1), (8, 16, 8, 128, 2), (0, 16, 8, 128, 1)):
        assert lib.kv_pool_create(*args, FAKE_K, FAKE_V, ctypes.byref(h)) == -1
    assert lib.kv_pool_create(8, 16, 8, 128, 1, FAKE_K + 8, FAKE_V, ctypes.byref(h)) == -1
    assert lib.kv_pool_create(8, 16, 8, 128, 1, None, FAKE_V, ctypes.byref(h)) == -1


def test_alloc_free_cycle_and_exhaustion(kp):
    p = _pool(kp, 8)
    try:
        assert kp.kv_pool_num_free(p) == 8
        a = kp.kv_block_alloc(p, 3)
        assert list(a) == [0, 1, 2]
        assert kp.kv_pool_num_free(p) == 5
        assert all(kp.kv_block_refcount(p, i) == 1 for i in a)
        with pytest.raises(kp.KVPError) as e:
            kp.kv_block_alloc(p, 6)
        assert e.value.status == -2 and kp.kv_pool_num_free(p) == 5     # all-or-nothing
        kp.kv_block_free(p, a)
        assert kp.kv_pool_num_free(p) == 8
        # LIFO reuse: the last freed block comes back first
        assert list(kp.kv_block_alloc(p, 1)) == [2]
    finally:
        kp.kv_pool_destroy(p)


def test_shared_prefix_refcounts(kp):
    # Figure 11-4 of page "11.2 连续批处理与 PagedAttention": blocks 1 and 4 are shared by
    # two requests (refcount 2); freeing one request keeps them allocated.
    p = _pool(kp, 10)
    try:
        kp.kv_block_claim(p, [1, 4, 7, 2])        # request A
        kp.kv_block_ref(p, [1, 4])                # request B shares the two full blocks
        kp.kv_block_claim(p, [8])                 # B's own block
        assert [kp.kv_block_refcount(p, i) for i in (1, 4, 7, 2, 8)] == [2, 2, 1, 1, 1]
        kp.kv_block_free(p, [1, 4, 7, 2])         # A finishes
        assert [kp.kv_block_refcount(p, i) for i in (1, 4, 7, 2, 8)] == [1, 1, 0, 0, 1]
        assert kp.kv_pool_num_free(p) == 10 - 3
        kp.kv_block_free(p, [1, 4, 8])            # B finishes
        assert kp.kv_pool_num_free(p) == 10
    finally:
        kp.kv_pool_destroy(p)


def test_errors_change_nothing(kp):
    p = _pool(kp, 6)
    try:
        kp.kv_block_claim(p, [3])
        for bad in ([3], [9], [-1], [0, 0]):
            with pytest.raises(kp.KVPError) as e:
                kp.kv_block_claim(p, bad)
            assert e.value.status == -3
        with pytest.raises(kp.KVPError) as e:
            kp.kv_block_free(p, [3, 3])           # would go below zero
        assert e.value.status == -7
        with pytest.raises(kp.KVPError) as e:
            kp.kv_block_ref(p, [3, 5])            # 5 is free
        assert e.value.status == -7
        assert kp.kv_block_refcount(p, 3) == 1 and kp.kv_pool_num_free(p) == 5
        with pytest.raises(kp.KVPError):
            kp.kv_block_free(p, [5])              # double free of a free block
        assert kp.kv_pool_num_free(p) == 5
    finally:
        kp.kv_pool_destroy(p)


def test_claim_then_alloc_never_hands_out_claimed(kp):
    rng = np.random.default_rng(0)
    p = _pool(kp, 64)
    try:
        claimed = rng.permutation(64)[:40]
        kp.kv_block_claim(p, claimed)
        rest = kp.kv_block_alloc(p, 24)
        assert sorted(set(rest) | set(claimed)) == list(range(64))
        with pytest.raises(kp.KVPError):
            kp.kv_block_alloc(p, 1)
    finally:
        kp.kv_pool_destroy(p)


def test_workspace_size_and_split_setting(kp):
    p = _pool(kp, 8)
    try:
        small = kp.paged_attention_workspace_size(p, 3, 7, 7)
        big = kp.paged_attention_workspace_size(p, 300, 8224, 8192)
        assert 0 < small < big and small % 256 == 0
        kp.kv_pool_set_decode_ctas(p, 5)
        assert kp.paged_attention_workspace_size(p, 300, 8224, 8192) == big
        for bad in (-1, 1025):
            with pytest.raises(kp.KVPError):
                kp.kv_pool_set_decode_ctas(p, bad)
        assert kp.lib.paged_attention_workspace_size(p, 3, 7, 16, 7) == 0     # only 32 query heads
        kp.kv_pool_set_nvtx(p, True)           # NVTX ranges: a host-side switch, no device work
        kp.kv_pool_set_nvtx(p, False)
        assert kp.lib.kv_pool_set_nvtx(None, 1) == -1
        kp.kv_pool_set_step_kernel(p, True)    # the mixed step kernel: a host-side switch too
        kp.kv_pool_set_step_kernel(p, False)
        for bad in (-1, 2):
            assert kp.lib.kv_pool_set_step_kernel(p, bad) == -1
        assert kp.lib.kv_pool_set_step_kernel(None, 1) == -1
        assert kp.paged_attention_workspace_size(p, 300, 8224, 8192) == big
    finally:
        kp.kv_pool_destroy(p)


def test_status_strings(kp):
    for code in kp.STATUS_NAMES:
        assert kp.lib.kvp_status_string(code)


def test_cow_and_swap_host_checks(kp):
    """The host-side rules of copy-on-write and swap (nothing here reaches a device)."""
    h = kp.kv_pool_create(FAKE_K, FAKE_V, num_blocks=8)
    try:
        a = [int(b) for b in kp.kv_block_alloc(h, 6)]
        # blocks nobody shares come back as they are, with nothing launched
        assert kp.kv_block_cow(h, a[:3]).tolist() == a[:3]
        assert [kp.kv_block_refcount(h, b) for b in a[:3]] == [1, 1, 1]
        # free or out-of-range sources
        free = [b for b in range(8) if b not in a]
        for bad in ([free[0]], [8], [-1]):
            with pytest.raises(kp.KVPError) as e:
                kp.kv_block_cow(h, bad)
            assert e.value.status == -3
        # three copies needed, two free blocks: refused, nothing changes
        kp.kv_block_ref(h, [a[0], a[1], a[2]])
        with pytest.raises(kp.KVPError) as e:
            kp.kv_block_cow(h, [a[0], a[1], a[2]])
        assert e.value.status == -2
        assert kp.kv_pool_num_free(h) == 2 and [kp.kv_block_refcount(h, b) for b in a[:3]] == [2, 2, 2]
        # swap: release checks first, then the host buffers must be page-locked memory
        import torch
        buf = torch.empty(4 * kp.BLOCK_BYTES, dtype=torch.uint8)       # pageable
        with pytest.raises(ValueError):
            kp.kv_blocks_swap_out(h, [a[3]], buf, buf)
        st = kp.lib.kv_blocks_swap_out(h, 1, (ctypes.c_int32 * 1)(free[0]), buf.data_ptr(), buf.data_ptr(), None)
        assert st == -7                                               # a free block
        st = kp.lib.kv_blocks_swap_out(h, 1, (ctypes.c_int32 * 1)(a[3]), buf.data_ptr(), buf.data_ptr(), None)
        assert st == -1 and kp.kv_block_refcount(h, a[3]) == 1         # pageable: refused, unchanged
        out = (ctypes.c_int32 * 3)()
        assert kp.lib.kv_blocks_swap_in(h, 3, buf.data_ptr(), buf.data_ptr(), out, None) == -2
        assert kp.lib.kv_blocks_swap_in(h, 1, buf.data_ptr(), buf.data_ptr(), out, None) == -1
        assert kp.kv_pool_num_free(h) == 2
    finally:
        kp.kv_pool_destroy(h)
