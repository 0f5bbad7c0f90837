// kv_append: scatter this step's new K/V rows into the block-paged cache.
//
// Address mapping of page "连续批处理与 PagedAttention 原理", section "block table 与地址
// 映射": position p of request r lives in physical block b = table[r][p / 16] at token
// offset p % 16.  The pool keeps each (block, KV head) tile of 16 x 128 bf16 contiguous,
// so one (row, head) write is a single 256-byte run: 16 lanes each store 16 bytes.
//
// One CTA of 256 threads per packed row: the threads first look the row's request up in
// cu_seqlens together (one round of loads instead of a serial binary search), then
// threads 0..127 move K and 128..255 move V; within each half, thread t handles head
// t / 16 and 16-byte chunk t % 16.  Loads of the new row are fully coalesced (2 KiB per
// tensor per row); stores are 256-byte runs per head.
#include "kvp_device.cuh"
#include "kvp_launch.h"

namespace kvp {

__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k_new,
                                                        const uint4* __restrict__ v_new,
                                                        const int32_t* __restrict__ cu,
                                                        const int32_t* __restrict__ ctx,
                                                        const int32_t* __restrict__ tables, int max_blocks,
                                                        int num_reqs, uint4* __restrict__ k_cache,
                                                        uint4* __restrict__ v_cache,
                                                        const int32_t* __restrict__ refcnt, int num_blocks,
                                                        uint32_t* __restrict__ err) {
    __shared__ long long s_dst;  // element-chunk index of (block, head 0, slot) or -1
    __shared__ int s_req;
    grid_dep_launch();   // the step's metadata kernel does not read the pool
    const int i = blockIdx.x;
    if (threadIdx.x == 0) s_req = -1;
    __syncthreads();
    // request r with cu[r] <= i < cu[r+1]: all threads test requests in parallel
    for (int r = threadIdx.x; r < num_reqs; r += blockDim.x)
        if (cu[r] <= i && i < cu[r + 1]) s_req = r;
    __syncthreads();
    if (threadIdx.x == 0) {
        long long dst = -1;
        const int r = s_req;
        if (r < 0) {
            raise_error(err, kErrBadMeta);
        } else {
            const int cl = ctx[r];
            const long long p = (long long)cl + (i - cu[r]);
            const long long lb = p >> 4;
            if (cl < 0 || lb >= max_blocks) {
                raise_error(err, kErrBadMeta);
            } else {
                const int b = tables[(size_t)r * max_blocks + lb];
                if (b < 0 || b >= num_blocks) {
                    raise_error(err, kErrBadBlock);
                } else {
                    const int rc = refcnt[b];
                    if (rc == 1) {
                        dst = ((long long)b * kNumKvHeads * kBlockSize + (p & 15)) * (kHeadBytes / 16);
                    } else {
                        raise_error(err, rc == 0 ? kErrBadBlock : kErrSharedWrite);
                    }
                }
            }
        }
        s_dst = dst;
    }
    __syncthreads();
    const long long dst = s_dst;
    if (dst < 0) return;
    const int t = threadIdx.x & 127;
    const int h = t >> 4, chunk = t & 15;
    const size_t src = (size_t)i * (kKvRowElems * 2 / 16) + h * (kHeadBytes / 16) + chunk;
    // (block, head h, slot) tile offset: head stride is 16 slots of 256 bytes
    const size_t d = (size_t)dst + (size_t)h * kBlockSize * (kHeadBytes / 16) + chunk;
    if (threadIdx.x < 128) {
        k_cache[d] = k_new[src];
    } else {
        v_cache[d] = v_new[src];
    }
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, const int32_t* cu, const int32_t* ctx,
                             const int32_t* tables, int max_blocks, int num_reqs, int num_tokens, void* k_cache,
                             void* v_cache, const int32_t* refcnt, int num_blocks, uint32_t* err,
                             cudaStream_t stream) {
    if (num_tokens <= 0) return cudaSuccess;
    kv_append_kernel<<<num_tokens, 256, 0, stream>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), cu, ctx, tables, max_blocks, num_reqs,
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), refcnt, num_blocks, err);
    return cudaGetLastError();
}

}  // namespace kvp
