// C-ABI entry points of libkvpaged: the block pool (free list + refcounts, the block
// manager of page "连续批处理与 PagedAttention 原理", section "块管理器"), kv_append and
// paged_attention_step.  Host code only; kernels live in the other .cu files.
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "kvpaged.h"
#include "kvp_device.cuh"
#include "kvp_launch.h"

namespace kvp {
cudaError_t configure_decode_kernel();
cudaError_t configure_prefill_kernel();
cudaError_t configure_mixed_kernel();
}  // namespace kvp

struct kvp_pool {
    int num_blocks = 0;
    void* k_cache = nullptr;
    void* v_cache = nullptr;
    std::vector<int32_t> free_list;  // stack; back() is handed out next
    std::vector<int32_t> free_pos;   // index in free_list, -1 when allocated
    std::vector<int32_t> refcnt;
    int dirty_lo = 1, dirty_hi = 0;  // refcount range changed since the last upload
    int decode_ctas = 0;  // 0: one decode CTA per SM
    int step_kernel = 0;  // 1: the mixed step kernel instead of the decode + prefill kernels
    // device state (made on first device call)
    int device = -1;
    int num_sms = 0;
    int32_t* d_refcnt = nullptr;
    uint32_t* d_err = nullptr;
    int32_t* h_stage[2] = {nullptr, nullptr};  // pinned staging for refcount uploads
    cudaEvent_t stage_ev[2] = {nullptr, nullptr};
    int stage_next = 0;
    CUtensorMap tmap_k;       // (block, head) tiles: boxes of 16 rows (prefill)
    CUtensorMap tmap_v;
    CUtensorMap tmap_k_blk;   // whole blocks: boxes of 128 rows (decode)
    CUtensorMap tmap_v_blk;
    // diagnostics
    int nvtx = 0;   // NVTX ranges around the library's calls and launches (off by default)
    long long launches = 0;
    std::vector<cudaEvent_t> t_events;  // 2 per timed launch
    std::vector<int> t_kind;
    int t_used = 0;
};

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

void mark_dirty(kvp_pool* p, int id) {
    if (p->dirty_lo > p->dirty_hi) {
        p->dirty_lo = p->dirty_hi = id;
    } else {
        p->dirty_lo = std::min(p->dirty_lo, id);
        p->dirty_hi = std::max(p->dirty_hi, id);
    }
}

// K or V pool viewed as rows of 128 bf16: row (b * 8 + h) * 16 + slot; boxes of 64 dims x
// box_rows rows (16: one (block, head) tile half; 128: one block's half), 128-byte swizzle.
bool encode_pool_map(CUtensorMap* m, void* base, int num_blocks, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kvp::kHeadDim, (cuuint64_t)num_blocks * kvp::kNumKvHeads * kvp::kBlockSize};
    const cuuint64_t strides[1] = {(cuuint64_t)kvp::kHeadBytes};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q [T][32 heads][128] viewed 3-D (dim, head, token); boxes of 64 dims x 4 heads (one KV
// group) x 32 tokens: 128 rows of 128 bytes, row = 4 * token + head, 128-byte swizzle.
bool encode_q_map(CUtensorMap* m, const void* q, int num_tokens) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kvp::kHeadDim, (cuuint64_t)kvp::kNumQHeads, (cuuint64_t)num_tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)kvp::kHeadBytes, (cuuint64_t)kvp::kQRowElems * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)kvp::kGroup, (cuuint32_t)kvp::kPrefillMmaTokens};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

void free_timing(kvp_pool* p) {
    for (cudaEvent_t e : p->t_events) cudaEventDestroy(e);
    p->t_events.clear();
    p->t_kind.clear();
    p->t_used = 0;
}

void release_device(kvp_pool* p) {
    if (p->device < 0) return;
    int prev = -1;
    cudaGetDevice(&prev);
    cudaSetDevice(p->device);
    cudaDeviceSynchronize();
    cudaFree(p->d_refcnt);
    cudaFree(p->d_err);
    for (int i = 0; i < 2; ++i) {
        if (p->h_stage[i]) cudaFreeHost(p->h_stage[i]);
        if (p->stage_ev[i]) cudaEventDestroy(p->stage_ev[i]);
    }
    free_timing(p);
    if (prev >= 0) cudaSetDevice(prev);
    p->device = -1;
}

// Make the device-side state on the current device (first device call of the pool).
kvp_status ensure_device(kvp_pool* p) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVP_E_CUDA;
    if (p->device >= 0) return p->device == dev ? KVP_OK : KVP_E_INVALID_ARG;
    p->device = dev;
    const size_t nb = (size_t)p->num_blocks;
    bool ok = cudaMalloc(&p->d_refcnt, nb * sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&p->d_err, sizeof(uint32_t)) == cudaSuccess &&
              cudaMemset(p->d_err, 0, sizeof(uint32_t)) == cudaSuccess &&
              cudaMemcpy(p->d_refcnt, p->refcnt.data(), nb * sizeof(int32_t), cudaMemcpyHostToDevice) ==
                  cudaSuccess &&
              cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
    for (int i = 0; ok && i < 2; ++i)
        ok = cudaHostAlloc(reinterpret_cast<void**>(&p->h_stage[i]), nb * sizeof(int32_t), cudaHostAllocDefault) ==
                 cudaSuccess &&
             cudaEventCreateWithFlags(&p->stage_ev[i], cudaEventDisableTiming) == cudaSuccess;
    ok = ok && kvp::configure_decode_kernel() == cudaSuccess && kvp::configure_prefill_kernel() == cudaSuccess &&
         kvp::configure_mixed_kernel() == cudaSuccess;
    const int tile_rows = kvp::kBlockSize, block_rows = kvp::kBlockSize * kvp::kNumKvHeads;
    ok = ok && encode_pool_map(&p->tmap_k, p->k_cache, p->num_blocks, tile_rows) &&
         encode_pool_map(&p->tmap_v, p->v_cache, p->num_blocks, tile_rows) &&
         encode_pool_map(&p->tmap_k_blk, p->k_cache, p->num_blocks, block_rows) &&
         encode_pool_map(&p->tmap_v_blk, p->v_cache, p->num_blocks, block_rows);
    if (!ok) {
        release_device(p);
        return KVP_E_CUDA;
    }
    p->dirty_lo = 1;
    p->dirty_hi = 0;
    return KVP_OK;
}

// Send refcount changes to the device mirror, in stream order.
kvp_status upload_refcounts(kvp_pool* p, cudaStream_t stream) {
    if (p->dirty_lo > p->dirty_hi) return KVP_OK;
    const int slot = p->stage_next;
    if (cudaEventSynchronize(p->stage_ev[slot]) != cudaSuccess) return KVP_E_CUDA;
    const int lo = p->dirty_lo, n = p->dirty_hi - p->dirty_lo + 1;
    std::memcpy(p->h_stage[slot], p->refcnt.data() + lo, (size_t)n * sizeof(int32_t));
    if (cudaMemcpyAsync(p->d_refcnt + lo, p->h_stage[slot], (size_t)n * sizeof(int32_t), cudaMemcpyHostToDevice,
                        stream) != cudaSuccess ||
        cudaEventRecord(p->stage_ev[slot], stream) != cudaSuccess)
        return KVP_E_CUDA;
    p->stage_next ^= 1;
    p->dirty_lo = 1;
    p->dirty_hi = 0;
    return KVP_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// An NVTX range in the library's own domain ("kvpaged") for the lifetime of the object,
// when the pool has ranges switched on: a profiler's timeline then shows kv_append, the
// attention step and each kernel launch by name.  Without a profiler attached the NVTX
// calls do nothing.
class NvtxRange {
   public:
    NvtxRange(const kvp_pool* p, const char* name) : on_(p && p->nvtx) {
        if (!on_) return;
        static nvtxDomainHandle_t dom = nvtxDomainCreateA("kvpaged");
        dom_ = dom;
        nvtxEventAttributes_t ev = {};
        ev.version = NVTX_VERSION;
        ev.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
        ev.messageType = NVTX_MESSAGE_TYPE_ASCII;
        ev.message.ascii = name;
        nvtxDomainRangePushEx(dom_, &ev);
    }
    ~NvtxRange() {
        if (on_) nvtxDomainRangePop(dom_);
    }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;

   private:
    bool on_;
    nvtxDomainHandle_t dom_ = nullptr;
};

const char* kernel_name(int kind) {
    switch (kind) {
        case KVP_KERNEL_APPEND: return "kv_append_kernel";
        case KVP_KERNEL_PREP: return "step_prep_kernel";
        case KVP_KERNEL_PREFILL: return "prefill_kernel";
        case KVP_KERNEL_DECODE: return "decode_kernel";
        case KVP_KERNEL_BLOCKS: return "block_move_kernel";
        case KVP_KERNEL_COMBINE: return "combine_kernel";
        case KVP_KERNEL_MIXED: return "mixed_step_kernel";
    }
    return "kernel";
}

// Launch one kernel through `fn`, counting it and, when timing is on, bracketing it with
// the next pair of events.
template <class F>
cudaError_t timed_launch(kvp_pool* p, int kind, cudaStream_t s, F&& fn) {
    NvtxRange range(p, kernel_name(kind));
    const int slot = p->t_used;
    const bool timed = slot < (int)p->t_kind.size();
    if (timed && cudaEventRecord(p->t_events[2 * slot], s) != cudaSuccess) return cudaErrorUnknown;
    const cudaError_t e = fn();
    if (e != cudaSuccess) return e;
    ++p->launches;
    if (timed) {
        if (cudaEventRecord(p->t_events[2 * slot + 1], s) != cudaSuccess) return cudaErrorUnknown;
        p->t_kind[slot] = kind;
        p->t_used = slot + 1;
    }
    return cudaSuccess;
}

// Device address of page-locked host memory (cudaHostAlloc / cudaHostRegister), or
// false for any other pointer.
bool host_device_ptr(const void* h, void** d) {
    cudaPointerAttributes at;
    if (!h || cudaPointerGetAttributes(&at, h) != cudaSuccess) {
        cudaGetLastError();   // clear the sticky-free error of a failed query
        return false;
    }
    if (at.type != cudaMemoryTypeHost || !at.devicePointer) return false;
    *d = at.devicePointer;
    return aligned16(*d);
}

// Copy n whole blocks (K and V) in launches of up to kMoveChunk: a side with ids is a pool
// indexed by block id, a side without is a host buffer indexed by list position.
kvp_status move_blocks(kvp_pool* p, const void* src_k, const void* src_v, const int32_t* src_ids, void* dst_k,
                       void* dst_v, const int32_t* dst_ids, int n, cudaStream_t s) {
    static thread_local kvp::BlockMoveArgs a;   // 8 KiB of ids: kept off the stack
    for (int off = 0; off < n; off += kvp::kMoveChunk) {
        const int m = std::min(kvp::kMoveChunk, n - off);
        const size_t host_off = (size_t)off * kvp::kBlockBytes;
        a.n = m;
        a.src[0] = static_cast<const uint8_t*>(src_k) + (src_ids ? 0 : host_off);
        a.src[1] = static_cast<const uint8_t*>(src_v) + (src_ids ? 0 : host_off);
        a.dst[0] = static_cast<uint8_t*>(dst_k) + (dst_ids ? 0 : host_off);
        a.dst[1] = static_cast<uint8_t*>(dst_v) + (dst_ids ? 0 : host_off);
        a.src_ids_used = src_ids ? 1 : 0;
        a.dst_ids_used = dst_ids ? 1 : 0;
        if (src_ids) std::memcpy(a.src_ids, src_ids + off, (size_t)m * sizeof(int32_t));
        if (dst_ids) std::memcpy(a.dst_ids, dst_ids + off, (size_t)m * sizeof(int32_t));
        if (timed_launch(p, KVP_KERNEL_BLOCKS, s, [&] { return kvp::launch_block_move(a, s); }) != cudaSuccess)
            return KVP_E_CUDA;
    }
    return KVP_OK;
}

// The checks of kv_block_free: every id in range, no refcount driven below zero.
kvp_status check_release(const kvp_pool* p, int n, const int32_t* ids) {
    std::vector<int32_t> sorted(ids, ids + n);
    std::sort(sorted.begin(), sorted.end());
    for (int i = 0; i < n;) {
        const int32_t id = sorted[i];
        if (id < 0 || id >= p->num_blocks) return KVP_E_BAD_BLOCK;
        int k = i;
        while (k < n && sorted[k] == id) ++k;
        if (p->refcnt[id] < k - i) return KVP_E_REFCOUNT;
        i = k;
    }
    return KVP_OK;
}

}  // namespace

extern "C" {

kvp_status kv_pool_create(int num_blocks, int block_size, int n_kv_heads, int head_dim, int dtype, void* k_cache,
                          void* v_cache, kvp_pool** out) {
    if (!out) return KVP_E_INVALID_ARG;
    *out = nullptr;
    if (num_blocks <= 0 || num_blocks > (1 << 24) || block_size != kvp::kBlockSize ||
        n_kv_heads != kvp::kNumKvHeads || head_dim != kvp::kHeadDim || dtype != KVP_DTYPE_BF16 || !k_cache ||
        !v_cache || !aligned16(k_cache) || !aligned16(v_cache))
        return KVP_E_INVALID_ARG;
    kvp_pool* p = new (std::nothrow) kvp_pool();
    if (!p) return KVP_E_INVALID_ARG;
    p->num_blocks = num_blocks;
    p->k_cache = k_cache;
    p->v_cache = v_cache;
    p->free_list.resize(num_blocks);
    p->free_pos.resize(num_blocks);
    p->refcnt.assign(num_blocks, 0);
    for (int i = 0; i < num_blocks; ++i) {
        p->free_list[i] = num_blocks - 1 - i;  // block 0 is handed out first
        p->free_pos[num_blocks - 1 - i] = i;
    }
    *out = p;
    return KVP_OK;
}

kvp_status kv_pool_destroy(kvp_pool* pool) {
    if (!pool) return KVP_OK;
    release_device(pool);
    delete pool;
    return KVP_OK;
}

kvp_status kv_block_alloc(kvp_pool* p, int n, int32_t* out_ids) {
    if (!p || n < 0 || (n > 0 && !out_ids)) return KVP_E_INVALID_ARG;
    if ((size_t)n > p->free_list.size()) return KVP_E_NO_BLOCKS;
    for (int i = 0; i < n; ++i) {
        const int32_t id = p->free_list.back();
        p->free_list.pop_back();
        p->free_pos[id] = -1;
        p->refcnt[id] = 1;
        mark_dirty(p, id);
        out_ids[i] = id;
    }
    return KVP_OK;
}

kvp_status kv_block_claim(kvp_pool* p, int n, const int32_t* ids) {
    if (!p || n < 0 || (n > 0 && !ids)) return KVP_E_INVALID_ARG;
    std::vector<int32_t> sorted(ids, ids + n);
    std::sort(sorted.begin(), sorted.end());
    for (int i = 0; i < n; ++i) {
        const int32_t id = sorted[i];
        if (id < 0 || id >= p->num_blocks || p->free_pos[id] < 0 || (i > 0 && sorted[i - 1] == id))
            return KVP_E_BAD_BLOCK;
    }
    for (int i = 0; i < n; ++i) {
        const int32_t id = ids[i];
        const int32_t pos = p->free_pos[id];
        const int32_t last = p->free_list.back();
        p->free_list[pos] = last;
        p->free_pos[last] = pos;
        p->free_list.pop_back();
        p->free_pos[id] = -1;
        p->refcnt[id] = 1;
        mark_dirty(p, id);
    }
    return KVP_OK;
}

kvp_status kv_block_ref(kvp_pool* p, int n, const int32_t* ids) {
    if (!p || n < 0 || (n > 0 && !ids)) return KVP_E_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= p->num_blocks) return KVP_E_BAD_BLOCK;
        if (p->refcnt[ids[i]] <= 0) return KVP_E_REFCOUNT;
    }
    for (int i = 0; i < n; ++i) {
        p->refcnt[ids[i]] += 1;
        mark_dirty(p, ids[i]);
    }
    return KVP_OK;
}

kvp_status kv_block_free(kvp_pool* p, int n, const int32_t* ids) {
    if (!p || n < 0 || (n > 0 && !ids)) return KVP_E_INVALID_ARG;
    const kvp_status st = check_release(p, n, ids);
    if (st != KVP_OK) return st;
    for (int i = 0; i < n; ++i) {
        const int32_t id = ids[i];
        if (--p->refcnt[id] == 0) {
            p->free_pos[id] = (int32_t)p->free_list.size();
            p->free_list.push_back(id);
        }
        mark_dirty(p, id);
    }
    return KVP_OK;
}

kvp_status kv_block_cow(kvp_pool* p, int n, const int32_t* src_ids, int32_t* out_ids, kvp_stream stream) {
    if (!p || n < 0 || (n > 0 && (!src_ids || !out_ids))) return KVP_E_INVALID_ARG;
    // decide every copy first (a block listed twice is shared by one fewer reference the
    // second time), so that nothing changes when a check fails
    std::unordered_map<int32_t, int> taken;
    std::vector<char> copy(n, 0);
    int copies = 0;
    for (int i = 0; i < n; ++i) {
        const int32_t id = src_ids[i];
        if (id < 0 || id >= p->num_blocks || p->refcnt[id] <= 0) return KVP_E_BAD_BLOCK;
        int& t = taken[id];
        if (p->refcnt[id] - t > 1) {
            copy[i] = 1;
            ++t;
            ++copies;
        }
    }
    if ((size_t)copies > p->free_list.size()) return KVP_E_NO_BLOCKS;
    if (copies > 0) {
        const kvp_status st = ensure_device(p);
        if (st != KVP_OK) return st;
    }
    std::vector<int32_t> srcs, dsts;
    srcs.reserve(copies);
    dsts.reserve(copies);
    for (int i = 0; i < n; ++i) {
        const int32_t id = src_ids[i];
        if (!copy[i]) {
            out_ids[i] = id;
            continue;
        }
        const int32_t nb = p->free_list.back();
        p->free_list.pop_back();
        p->free_pos[nb] = -1;
        p->refcnt[nb] = 1;
        p->refcnt[id] -= 1;
        mark_dirty(p, nb);
        mark_dirty(p, id);
        out_ids[i] = nb;
        srcs.push_back(id);
        dsts.push_back(nb);
    }
    return move_blocks(p, p->k_cache, p->v_cache, srcs.data(), p->k_cache, p->v_cache, dsts.data(), copies,
                       reinterpret_cast<cudaStream_t>(stream));
}

kvp_status kv_blocks_swap_out(kvp_pool* p, int n, const int32_t* ids, void* host_k, void* host_v,
                              kvp_stream stream) {
    if (!p || n < 0 || (n > 0 && !ids)) return KVP_E_INVALID_ARG;
    if (n == 0) return KVP_OK;
    kvp_status st = check_release(p, n, ids);
    if (st != KVP_OK) return st;
    void *dk = nullptr, *dv = nullptr;
    if (!host_device_ptr(host_k, &dk) || !host_device_ptr(host_v, &dv)) return KVP_E_INVALID_ARG;
    if ((st = ensure_device(p)) != KVP_OK) return st;
    st = move_blocks(p, p->k_cache, p->v_cache, ids, dk, dv, nullptr, n, reinterpret_cast<cudaStream_t>(stream));
    if (st != KVP_OK) return st;
    return kv_block_free(p, n, ids);
}

kvp_status kv_blocks_swap_in(kvp_pool* p, int n, const void* host_k, const void* host_v, int32_t* out_ids,
                             kvp_stream stream) {
    if (!p || n < 0 || (n > 0 && !out_ids)) return KVP_E_INVALID_ARG;
    if (n == 0) return KVP_OK;
    if ((size_t)n > p->free_list.size()) return KVP_E_NO_BLOCKS;
    void *dk = nullptr, *dv = nullptr;
    if (!host_device_ptr(host_k, &dk) || !host_device_ptr(host_v, &dv)) return KVP_E_INVALID_ARG;
    kvp_status st = ensure_device(p);
    if (st != KVP_OK) return st;
    if ((st = kv_block_alloc(p, n, out_ids)) != KVP_OK) return st;
    return move_blocks(p, dk, dv, nullptr, p->k_cache, p->v_cache, out_ids, n, reinterpret_cast<cudaStream_t>(stream));
}

int kv_pool_num_free(const kvp_pool* p) { return p ? (int)p->free_list.size() : -1; }

int kv_block_refcount(const kvp_pool* p, int32_t id) {
    if (!p || id < 0 || id >= p->num_blocks) return -1;
    return p->refcnt[id];
}

kvp_status kv_pool_set_nvtx(kvp_pool* p, int on) {
    if (!p) return KVP_E_INVALID_ARG;
    p->nvtx = on ? 1 : 0;
    return KVP_OK;
}

kvp_status kv_pool_set_step_kernel(kvp_pool* p, int mixed) {
    if (!p || (mixed != 0 && mixed != 1)) return KVP_E_INVALID_ARG;
    p->step_kernel = mixed;
    return KVP_OK;
}

kvp_status kv_pool_set_decode_ctas(kvp_pool* p, int ctas) {
    if (!p || ctas < 0 || ctas > kvp::kMaxDecodeCtas) return KVP_E_INVALID_ARG;
    p->decode_ctas = ctas;
    return KVP_OK;
}

kvp_status kv_append(kvp_pool* p, const void* k_new, const void* v_new, const int32_t* cu_seqlens_q,
                     const int32_t* context_lens, const int32_t* block_tables, int max_blocks_per_seq, int num_reqs,
                     int num_tokens, kvp_stream stream) {
    if (!p || num_tokens < 0 || num_reqs < 0) return KVP_E_INVALID_ARG;
    if (num_tokens == 0) return KVP_OK;
    if (num_reqs < 1 || max_blocks_per_seq < 1 || !k_new || !v_new || !cu_seqlens_q || !context_lens ||
        !block_tables || !aligned16(k_new) || !aligned16(v_new))
        return KVP_E_INVALID_ARG;
    NvtxRange range(p, "kv_append");
    kvp_status st = ensure_device(p);
    if (st != KVP_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((st = upload_refcounts(p, s)) != KVP_OK) return st;
    const cudaError_t e = timed_launch(p, KVP_KERNEL_APPEND, s, [&] {
        return kvp::launch_kv_append(k_new, v_new, cu_seqlens_q, context_lens, block_tables, max_blocks_per_seq,
                                     num_reqs, num_tokens, p->k_cache, p->v_cache, p->d_refcnt, p->num_blocks,
                                     p->d_err, s);
    });
    return e == cudaSuccess ? KVP_OK : KVP_E_CUDA;
}

size_t paged_attention_workspace_size(const kvp_pool* p, int num_reqs, int num_tokens, int n_q_heads,
                                      int max_context_len) {
    if (!p || num_reqs < 0 || num_tokens < 0 || max_context_len < 0 || n_q_heads != kvp::kNumQHeads) return 0;
    return kvp::make_step_layout(num_reqs, num_tokens).total;
}

kvp_status paged_attention_step(kvp_pool* p, const void* q, void* out, const int32_t* cu_seqlens_q,
                                const int32_t* context_lens, const int32_t* block_tables, int max_blocks_per_seq,
                                int num_reqs, int num_tokens, int n_q_heads, int max_q_len, int max_context_len,
                                float softmax_scale, void* workspace, size_t workspace_bytes, kvp_stream stream) {
    if (!p || num_tokens < 0 || num_reqs < 0 || n_q_heads != kvp::kNumQHeads) return KVP_E_INVALID_ARG;
    if (num_tokens == 0) return KVP_OK;
    if (num_reqs < 1 || max_blocks_per_seq < 1 || max_q_len < 1 || max_context_len < 0 || !q || !out ||
        !cu_seqlens_q || !context_lens || !block_tables || !aligned16(q) || !aligned16(out) ||
        !(softmax_scale > 0.f))
        return KVP_E_INVALID_ARG;
    kvp::StepLayout lay = kvp::make_step_layout(num_reqs, num_tokens);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < lay.total)
        return KVP_E_WORKSPACE;
    NvtxRange range(p, "paged_attention_step");
    kvp_status st = ensure_device(p);
    if (st != KVP_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    kvp::StepArgs a;
    a.q = q;
    a.out = out;
    a.cu_seqlens_q = cu_seqlens_q;
    a.context_lens = context_lens;
    a.block_tables = block_tables;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_reqs = num_reqs;
    a.num_tokens = num_tokens;
    a.max_q_len = max_q_len;
    a.max_context_len = max_context_len;
    a.softmax_scale = softmax_scale;
    a.k_cache = p->k_cache;
    a.v_cache = p->v_cache;
    a.num_blocks = p->num_blocks;
    a.err = p->d_err;
    a.ws = static_cast<char*>(workspace);
    a.lay = lay;
    a.num_sms = p->num_sms;
    a.decode_ctas = p->decode_ctas;
    if (timed_launch(p, KVP_KERNEL_PREP, s, [&] { return kvp::launch_step_prep(a, s); }) != cudaSuccess)
        return KVP_E_CUDA;
    if (p->step_kernel == 1) {
        // one grid for the decode rows and the prefill tiles (work tickets)
        CUtensorMap tq;
        if (!encode_q_map(&tq, q, num_tokens)) return KVP_E_CUDA;
        if (timed_launch(p, KVP_KERNEL_MIXED, s, [&] {
                return kvp::launch_mixed(a, &tq, &p->tmap_k, &p->tmap_v, &p->tmap_k_blk, &p->tmap_v_blk, s);
            }) != cudaSuccess)
            return KVP_E_CUDA;
    } else {
        // decode first; the prefill kernel follows as its programmatic dependent and runs on
        // the SMs the decode leaves free (the metadata kernel sizes the split)
        if (timed_launch(p, KVP_KERNEL_DECODE, s,
                         [&] { return kvp::launch_decode(a, &p->tmap_k_blk, &p->tmap_v_blk, s); }) != cudaSuccess)
            return KVP_E_CUDA;
        if (max_q_len >= 2 && lay.max_prefill_tiles > 0) {
            CUtensorMap tq;
            if (!encode_q_map(&tq, q, num_tokens)) return KVP_E_CUDA;
            if (timed_launch(p, KVP_KERNEL_PREFILL, s,
                             [&] { return kvp::launch_prefill(a, &tq, &p->tmap_k, &p->tmap_v, s); }) != cudaSuccess)
                return KVP_E_CUDA;
        }
    }
    if (timed_launch(p, KVP_KERNEL_COMBINE, s, [&] { return kvp::launch_combine(a, s); }) != cudaSuccess)
        return KVP_E_CUDA;
    return KVP_OK;
}

kvp_status kv_pool_get_error(kvp_pool* p, kvp_stream stream, uint32_t* bits) {
    if (bits) *bits = 0;
    if (!p) return KVP_E_INVALID_ARG;
    if (p->device < 0) return KVP_OK;  // nothing ran on a device yet
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t w = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpyAsync(&w, p->d_err, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(p->d_err, 0, sizeof(uint32_t), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return KVP_E_CUDA;
    if (bits) *bits = w;
    if (w & KVP_ERRBIT_BAD_BLOCK) return KVP_E_BAD_BLOCK;
    if (w & KVP_ERRBIT_SHARED_WRITE) return KVP_E_SHARED_WRITE;
    if (w & KVP_ERRBIT_BAD_META) return KVP_E_BAD_META;
    if (w & KVP_ERRBIT_TIMEOUT) return KVP_E_TIMEOUT;
    return KVP_OK;
}

kvp_status kv_pool_enable_timing(kvp_pool* p, int max_launches) {
    if (!p || max_launches < 0) return KVP_E_INVALID_ARG;
    if (max_launches > 0) {
        kvp_status st = ensure_device(p);
        if (st != KVP_OK) return st;
    }
    if (p->device >= 0) {
        int prev = -1;
        cudaGetDevice(&prev);
        cudaSetDevice(p->device);
        cudaDeviceSynchronize();
        free_timing(p);
        bool ok = true;
        p->t_events.resize(2 * (size_t)max_launches, nullptr);
        for (auto& e : p->t_events) ok = ok && cudaEventCreate(&e) == cudaSuccess;
        p->t_kind.assign(max_launches, -1);
        if (prev >= 0) cudaSetDevice(prev);
        if (!ok) {
            free_timing(p);
            return KVP_E_CUDA;
        }
    }
    return KVP_OK;
}

kvp_status kv_pool_read_timing(kvp_pool* p, int* counts, float* ms) {
    if (!p || !counts || !ms) return KVP_E_INVALID_ARG;
    for (int k = 0; k < KVP_NUM_KERNELS; ++k) {
        counts[k] = 0;
        ms[k] = 0.f;
    }
    if (p->t_used > 0 && cudaEventSynchronize(p->t_events[2 * p->t_used - 1]) != cudaSuccess) return KVP_E_CUDA;
    for (int i = 0; i < p->t_used; ++i) {
        float t = 0.f;
        if (cudaEventElapsedTime(&t, p->t_events[2 * i], p->t_events[2 * i + 1]) != cudaSuccess) return KVP_E_CUDA;
        counts[p->t_kind[i]] += 1;
        ms[p->t_kind[i]] += t;
    }
    p->t_used = 0;
    return KVP_OK;
}

long long kv_pool_launch_count(const kvp_pool* p) { return p ? p->launches : -1; }

}  // extern "C"

namespace kvp {
// Device the pool's device-side state lives on, or -1 if it has none yet.
int pool_device(const kvp_pool* p) { return p ? p->device : -1; }
}  // namespace kvp

extern "C" {

const char* kvp_status_string(kvp_status s) {
    switch (s) {
        case KVP_OK: return "ok";
        case KVP_E_INVALID_ARG: return "invalid argument";
        case KVP_E_NO_BLOCKS: return "no free blocks";
        case KVP_E_BAD_BLOCK: return "bad block id";
        case KVP_E_SHARED_WRITE: return "write into a shared block";
        case KVP_E_BAD_META: return "inconsistent step metadata";
        case KVP_E_CUDA: return "CUDA runtime error";
        case KVP_E_REFCOUNT: return "refcount underflow (double free)";
        case KVP_E_WORKSPACE: return "workspace missing or too small";
        case KVP_E_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

}  // extern "C"
