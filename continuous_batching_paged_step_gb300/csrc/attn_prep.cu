// Step metadata: turn cu_seqlens_q / context_lens into work lists for the attention
// kernels, on the device (the packed layout of page "Continuous Batching 深入实现",
// section "方案：Ragged Batch + cu_seqlens": each request's rows are a contiguous range
// of the flat token matrix, delimited by cu_seqlens).
//
// Request r brings q_r = cu[r+1] - cu[r] rows at positions ctx_r .. ctx_r + q_r - 1.
//   q_r == 1 (decode): its history of ctx_r + 1 keys (ceil((ctx_r+1)/16) blocks) is cut
//     into chunks of `chunk_pages` blocks; one decode work item per chunk.  With more
//     than one chunk the items write split-KV partials and a combine entry merges them.
//   q_r >= 2 (prefill chunk): one tile per 32 query tokens (x 4 query heads of a KV group
//     = 128 MMA rows), emitted last tile first so the longest tiles start earliest.
// One CTA of 1024 threads scans the requests in rounds of 1024 (block-wide exclusive
// scan of four counts).  Inconsistent metadata sets KVP_ERRBIT_BAD_META; a request that
// fails its own checks gets no work, and a cu_seqlens array that is not a monotone map
// of [0, num_tokens] gets no work at all.
#include "kvp_device.cuh"
#include "kvp_launch.h"

namespace kvp {

namespace {

constexpr int kPrepThreads = 1024;

__device__ __forceinline__ int4 warp_incl_scan(int4 v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int4 u;
        u.x = __shfl_up_sync(0xffffffffu, v.x, o);
        u.y = __shfl_up_sync(0xffffffffu, v.y, o);
        u.z = __shfl_up_sync(0xffffffffu, v.z, o);
        u.w = __shfl_up_sync(0xffffffffu, v.w, o);
        if (lane >= o) {
            v.x += u.x;
            v.y += u.y;
            v.z += u.z;
            v.w += u.w;
        }
    }
    return v;
}

__global__ void __launch_bounds__(kPrepThreads) step_prep_kernel(
    const int32_t* __restrict__ cu, const int32_t* __restrict__ ctx, int num_reqs, int num_tokens,
    int max_q_len, int max_context_len, int max_blocks, int chunk_pages, int max_decode_items,
    int max_partials, int max_prefill_tiles, int max_combines, int32_t* __restrict__ counters,
    int4* __restrict__ dec_items, int4* __restrict__ pre_tiles, int4* __restrict__ combines,
    uint32_t* __restrict__ err) {
    __shared__ int s_ok;
    __shared__ int4 s_warp[32];
    __shared__ int4 s_base;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_ok = (cu[0] == 0 && cu[num_reqs] == num_tokens) ? 1 : 0;
        s_base = make_int4(0, 0, 0, 0);
    }
    __syncthreads();
    for (int r = tid; r < num_reqs; r += kPrepThreads)
        if (cu[r + 1] < cu[r]) s_ok = 0;
    __syncthreads();
    if (!s_ok) {
        if (tid == 0) {
            raise_error(err, kErrBadMeta);
            counters[0] = counters[1] = counters[2] = 0;
        }
        return;
    }
    for (int round = 0; round < num_reqs; round += kPrepThreads) {
        const int r = round + tid;
        // x: decode items, y: partial slots, z: prefill tiles, w: combine entries
        int4 n = make_int4(0, 0, 0, 0);
        int q = 0, c = 0, pages = 0;
        if (r < num_reqs) {
            q = cu[r + 1] - cu[r];
            c = ctx[r];
            const bool ok = c >= 0 && c <= max_context_len && q <= max_q_len &&
                            (long long)c + q <= (long long)max_blocks * kBlockSize;
            if (!ok) {
                if (q > 0) raise_error(err, kErrBadMeta);
            } else if (q == 1) {
                pages = (c + 1 + kBlockSize - 1) / kBlockSize;
                const int chunks = (pages + chunk_pages - 1) / chunk_pages;
                n.x = chunks;
                if (chunks > 1) {
                    n.y = chunks;
                    n.w = 1;
                }
            } else if (q > 1) {
                n.z = (q + kPrefillTileTokens - 1) / kPrefillTileTokens;
            }
        }
        const int4 incl = warp_incl_scan(n, lane);
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int4 wt = s_warp[lane];
            const int4 wi = warp_incl_scan(wt, lane);
            s_warp[lane] = make_int4(wi.x - wt.x, wi.y - wt.y, wi.z - wt.z, wi.w - wt.w);
        }
        __syncthreads();
        const int4 wex = s_warp[warp];
        const int4 base = s_base;
        const int dx = base.x + wex.x + incl.x - n.x;
        const int dy = base.y + wex.y + incl.y - n.y;
        const int dz = base.z + wex.z + incl.z - n.z;
        const int dw = base.w + wex.w + incl.w - n.w;
        if (n.x > 0) {
            if (dx + n.x > max_decode_items || dy + n.y > max_partials || dw + n.w > max_combines) {
                raise_error(err, kErrBadMeta);
            } else {
                for (int k = 0; k < n.x; ++k) {
                    const int first = k * chunk_pages;
                    const int np = min(chunk_pages, pages - first);
                    dec_items[dx + k] = make_int4(r, first, np, n.x > 1 ? dy + k : -1);
                }
                if (n.w) combines[dw] = make_int4(r, dy, n.x, 0);
            }
        }
        if (n.z > 0) {
            if (dz + n.z > max_prefill_tiles) {
                raise_error(err, kErrBadMeta);
            } else {
                for (int t = 0; t < n.z; ++t) {
                    const int tok0 = (n.z - 1 - t) * kPrefillTileTokens;
                    pre_tiles[dz + t] = make_int4(r, tok0, min(kPrefillTileTokens, q - tok0), 0);
                }
            }
        }
        __syncthreads();
        if (tid == kPrepThreads - 1) {
            const int4 tot = make_int4(dx + n.x, dy + n.y, dz + n.z, dw + n.w);
            s_base = tot;
        }
        __syncthreads();
    }
    if (tid == 0) {
        const int4 b = s_base;
        counters[0] = min(b.x, max_decode_items);
        counters[1] = min(b.z, max_prefill_tiles);
        counters[2] = min(b.w, max_combines);
    }
}

}  // namespace

StepLayout make_step_layout(int num_reqs, int num_tokens, int max_context_len, int chunk_pages) {
    StepLayout L{};
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const int dec_reqs = num_reqs < num_tokens ? num_reqs : num_tokens;
    const int max_pages = (max_context_len + 1 + kBlockSize - 1) / kBlockSize;
    const int max_chunks = (max_pages + chunk_pages - 1) / chunk_pages;
    const int pre_reqs = num_reqs < num_tokens / 2 ? num_reqs : num_tokens / 2;
    L.decode_chunk_pages = chunk_pages;
    L.max_decode_items = dec_reqs * max_chunks;
    L.max_partials = max_chunks > 1 ? dec_reqs * max_chunks : 0;
    L.max_combines = max_chunks > 1 ? dec_reqs : 0;
    L.max_prefill_tiles = num_tokens / kPrefillTileTokens + pre_reqs + 1;
    size_t off = 0;
    L.counters_off = off;
    off = up(off + 8 * sizeof(int32_t));
    L.decode_items_off = off;
    off = up(off + (size_t)L.max_decode_items * sizeof(int4));
    L.prefill_tiles_off = off;
    off = up(off + (size_t)L.max_prefill_tiles * sizeof(int4));
    L.combines_off = off;
    off = up(off + (size_t)L.max_combines * sizeof(int4));
    L.part_acc_off = off;
    off = up(off + (size_t)L.max_partials * kNumQHeads * kHeadDim * sizeof(float));
    L.part_ml_off = off;
    off = up(off + (size_t)L.max_partials * kNumQHeads * sizeof(float2));
    L.total = off;
    return L;
}

cudaError_t launch_step_prep(const StepArgs& a, cudaStream_t stream) {
    const StepLayout& L = a.lay;
    step_prep_kernel<<<1, kPrepThreads, 0, stream>>>(
        a.cu_seqlens_q, a.context_lens, a.num_reqs, a.num_tokens, a.max_q_len, a.max_context_len,
        a.max_blocks_per_seq, L.decode_chunk_pages, L.max_decode_items, L.max_partials, L.max_prefill_tiles,
        L.max_combines, reinterpret_cast<int32_t*>(a.ws + L.counters_off),
        reinterpret_cast<int4*>(a.ws + L.decode_items_off), reinterpret_cast<int4*>(a.ws + L.prefill_tiles_off),
        reinterpret_cast<int4*>(a.ws + L.combines_off), a.err);
    return cudaGetLastError();
}

}  // namespace kvp
