// kv_append: scatter this step's new K/V rows into the block-paged cache.
//
// Address mapping of page "连续批处理与 PagedAttention 原理", section "block table 与地址
// 映射": position p of request r lives in physical block b = table[r][p / 16] at token
// offset p % 16.  The pool keeps each (block, KV head) tile of 16 x 128 bf16 contiguous,
// so one (row, head) write is a single 256-byte run: 16 lanes each store 16 bytes.
//
// One warp per packed row (8 rows per CTA of 256 threads, so a whole step is one wave of
// CTAs).  The CTA first copies cu_seqlens and context_lens into shared memory (steps of
// up to 2,048 requests; larger ones search global memory); lane 0 of each warp then finds
// its row's request by binary search (cu_seqlens is monotone), checks the context
// length, the table entry and the block's refcount, and hands the
// destination to the warp; the 32 lanes then move the row's 2 KiB of K and 2 KiB of V, 16
// bytes each per pass, fully coalesced on the read side and in 256-byte runs per head
// (half a warp) on the write side.
#include "kvp_device.cuh"
#include "kvp_launch.h"

namespace kvp {

constexpr int kAppendRowsPerCta = 8;   // one warp per row
constexpr int kAppendSmemReqs = 2048;  // requests whose metadata a CTA stages in shared memory

__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k_new,
                                                        const uint4* __restrict__ v_new,
                                                        const int32_t* __restrict__ cu,
                                                        const int32_t* __restrict__ ctx,
                                                        const int32_t* __restrict__ tables, int max_blocks,
                                                        int num_reqs, int num_tokens, uint4* __restrict__ k_cache,
                                                        uint4* __restrict__ v_cache,
                                                        const int32_t* __restrict__ refcnt, int num_blocks,
                                                        uint32_t* __restrict__ err) {
    __shared__ int32_t s_cu[kAppendSmemReqs + 1];
    __shared__ int32_t s_ctx[kAppendSmemReqs];
    grid_dep_launch();   // the step's metadata kernel does not read the pool
    // Launched as a programmatic dependent of whatever precedes it in the stream (normally the
    // previous step's last kernel), so its CTAs are resident when that kernel ends; nothing is
    // read or written before that kernel has completed.
    grid_dep_wait();
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * kAppendRowsPerCta + (threadIdx.x >> 5);
    // The row's K and V first: their loads do not depend on where the row goes, so they
    // are in flight while the metadata below is looked up.
    constexpr int kRowChunks = kKvRowElems * 2 / 16;   // 128 chunks of 16 bytes per row and tensor
    constexpr int kLaneChunks = kRowChunks / 32;
    const size_t src = (size_t)i * kRowChunks;
    uint4 kv[kLaneChunks], vv[kLaneChunks];
    if (i < num_tokens) {
#pragma unroll
        for (int k = 0; k < kLaneChunks; ++k) {
            kv[k] = k_new[src + k * 32 + lane];
            vv[k] = v_new[src + k * 32 + lane];
        }
    }
    const bool staged = num_reqs <= kAppendSmemReqs;
    if (staged) {
        for (int k = threadIdx.x; k <= num_reqs; k += blockDim.x) s_cu[k] = cu[k];
        for (int k = threadIdx.x; k < num_reqs; k += blockDim.x) s_ctx[k] = ctx[k];
        __syncthreads();
    }
    const int32_t* cu_r = staged ? s_cu : cu;
    const int32_t* ctx_r = staged ? s_ctx : ctx;
    if (i >= num_tokens) return;
    long long dst = -1;   // element-chunk index of (block, head 0, slot), or -1
    if (lane == 0) {
        // the last request r with cu[r] <= i; the row belongs to it iff i < cu[r + 1]
        int a = 0, b = num_reqs - 1;
        while (a < b) {
            const int mid = (a + b + 1) >> 1;
            if (cu_r[mid] <= i) a = mid;
            else b = mid - 1;
        }
        const int r = a;
        if (!(cu_r[r] <= i && i < cu_r[r + 1])) {
            raise_error(err, kErrBadMeta);
        } else {
            const int cl = ctx_r[r];
            const long long p = (long long)cl + (i - cu_r[r]);
            const long long lb = p >> 4;
            if (cl < 0 || lb >= max_blocks) {
                raise_error(err, kErrBadMeta);
            } else {
                const int bid = tables[(size_t)r * max_blocks + lb];
                if (bid < 0 || bid >= num_blocks) {
                    raise_error(err, kErrBadBlock);
                } else {
                    const int rc = refcnt[bid];
                    if (rc == 1) {
                        dst = ((long long)bid * kNumKvHeads * kBlockSize + (p & 15)) * (kHeadBytes / 16);
                    } else {
                        raise_error(err, rc == 0 ? kErrBadBlock : kErrSharedWrite);
                    }
                }
            }
        }
    }
    dst = __shfl_sync(0xffffffffu, dst, 0);
    if (dst < 0) return;
#pragma unroll
    for (int k = 0; k < kLaneChunks; ++k) {
        const int j = k * 32 + lane;
        const int h = j >> 4, chunk = j & 15;
        // (block, head h, slot) tile offset: head stride is 16 slots of 256 bytes
        const size_t d = (size_t)dst + (size_t)h * kBlockSize * (kHeadBytes / 16) + chunk;
        k_cache[d] = kv[k];
        v_cache[d] = vv[k];
    }
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, const int32_t* cu, const int32_t* ctx,
                             const int32_t* tables, int max_blocks, int num_reqs, int num_tokens, void* k_cache,
                             void* v_cache, const int32_t* refcnt, int num_blocks, uint32_t* err,
                             cudaStream_t stream) {
    if (num_tokens <= 0) return cudaSuccess;
    const int grid = (num_tokens + kAppendRowsPerCta - 1) / kAppendRowsPerCta;
    return launch_pdl(kv_append_kernel, dim3(grid), dim3(256), 0, stream, static_cast<const uint4*>(k_new),
                      static_cast<const uint4*>(v_new), cu, ctx, tables, max_blocks, num_reqs, num_tokens,
                      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), refcnt, num_blocks, err);
}

}  // namespace kvp
