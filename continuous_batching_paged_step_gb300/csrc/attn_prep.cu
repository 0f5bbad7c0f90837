// Step metadata: turn cu_seqlens_q / context_lens into work descriptions for the
// attention kernels, on the device (the packed layout of page "Continuous Batching 深入
// 实现", section "方案：Ragged Batch + cu_seqlens": each request's rows are a contiguous
// range of the flat token matrix, delimited by cu_seqlens).
//
// Request r brings q_r = cu[r+1] - cu[r] rows at positions ctx_r .. ctx_r + q_r - 1.
//   q_r == 1 (decode): its history of ctx_r + 1 keys covers ceil((ctx_r+1)/16) blocks;
//     page_off[r] is the exclusive prefix sum of those block counts over the requests
//     (0 blocks for other requests), page_off[num_reqs] the total.  The decode kernel
//     shares the total out among its CTAs; counters[4] (zeroed here) counts the chunks
//     of their ranges' tails the decode CTAs have taken.
//   q_r >= 2 (prefill chunk): one tile per 64 query tokens (two MMA tiles of 32 tokens x
//     4 query heads of a KV group).  The tiles of all chunks are emitted longest first
//     (by the number of 128-key tiles their last row reads), so that the prefill kernel,
//     whose CTAs start in list order, ends on its shortest tiles: a chunk after a long
//     cached prefix would otherwise leave its 50-60-key-tile CTAs for last.  The order
//     is a counting sort over key-tile counts; tiles with equal counts come in any order
//     (every tile writes only its own rows).
// SM split: the decode rows are HBM-bound and the prefill tiles tensor-bound, so the
// attention kernels run side by side: the decode kernel takes counters[2] CTAs (one per
// SM) and leaves the other SMs to prefill tiles, which start while the decode runs.  The
// split follows a simple cost model (below) of the two kernels' work; counters[3] is the
// prefill kernel's exit count, zeroed here.
// One CTA of 1024 threads scans the requests in rounds of 1024 (block-wide exclusive
// scan).  Inconsistent metadata sets KVP_ERRBIT_BAD_META; a request that fails its own
// checks gets no work, and a cu_seqlens array that is not a monotone map of
// [0, num_tokens] gets no work at all.
#include "kvp_device.cuh"
#include "kvp_launch.h"

namespace kvp {

namespace {

constexpr int kPrepThreads = 1024;
constexpr int kTileBins = 1024;   // key-tile counts of prefill tiles (larger ones share the last bin)

// Key tiles (128 keys) read by the last row of the prefill tile of `ntok` tokens that
// starts `tok0` tokens into a chunk after `c` cached tokens, as a sort bin.
__device__ __forceinline__ int tile_bin(int c, int tok0, int ntok) {
    return min((c + tok0 + ntok - 1) / 128 + 1, kTileBins - 1);
}

// Cost model of the SM split.  Prefill work is counted in units of one key tile of one
// prefill CTA (128 keys x 64 query tokens x 4 heads through QK^T, softmax and P.V: about
// 2.2 us on a GB300 SM), plus a fixed start/finish per CTA.  The decode is HBM-bound: on
// enough SMs it streams its blocks (64 KiB of K and V each) at about 0.0102 us per block
// for the whole GPU, and a single SM streams about one block per 0.77 us.  So the decode
// keeps as many SMs as the prefill leaves it, where the prefill is given enough SMs to
// finish its work in about the decode's HBM-bound time (its tiles run about 1.5x slower
// beside a decode that saturates HBM); but never fewer SMs than it needs to finish
// within the prefill's own time on the whole GPU (x 1.25), up to the 64 SMs that keep
// HBM near its streaming rate.
constexpr float kUnitUs = 2.2f;
constexpr float kTileFixedUnits = 2.f;
constexpr float kDecodeBlockUsGpu = 0.0102f;
constexpr float kDecodeBlockUsSm = 0.77f;
constexpr float kPrefillBesideDecode = 1.5f;
constexpr float kDecodeMargin = 1.25f;
constexpr int kDecodeHbmSms = 64;

// Decode CTAs for P decode blocks next to prefill work w (units) on n SMs.
__device__ int decode_sm_share(int P, float w, int n) {
    if (P <= 0 || w <= 0.f || n < 2) return n;
    const float prefill_us = w * kUnitUs;                       // SM-microseconds
    const float decode_us = P * kDecodeBlockUsGpu;              // on the whole GPU
    const float n_p = ceilf(kPrefillBesideDecode * prefill_us / decode_us);
    const float lo = fminf(ceilf(kDecodeMargin * P * kDecodeBlockUsSm * n / prefill_us), (float)kDecodeHbmSms);
    const float d = fmaxf(lo, (float)n - n_p);
    return max(1, min(n - 1, (int)d));
}

__device__ __forceinline__ int2 warp_incl_scan(int2 v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int ux = __shfl_up_sync(0xffffffffu, v.x, o);
        const int uy = __shfl_up_sync(0xffffffffu, v.y, o);
        if (lane >= o) {
            v.x += ux;
            v.y += uy;
        }
    }
    return v;
}

__global__ void __launch_bounds__(kPrepThreads) step_prep_kernel(
    const int32_t* __restrict__ cu, const int32_t* __restrict__ ctx, int num_reqs, int num_tokens, int max_q_len,
    int max_context_len, int max_blocks, int max_prefill_tiles, int num_sms, int32_t* __restrict__ counters,
    int32_t* __restrict__ page_off, int4* __restrict__ pre_tiles,
    uint32_t* __restrict__ err) {
    __shared__ int s_ok;
    __shared__ int2 s_warp[32];
    __shared__ int2 s_base;
    __shared__ float s_w[32];
    __shared__ int s_hist[kTileBins];    // tiles per bin, then the bin's next output slot
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    grid_dep_launch();
    if (tid == 0) {
        s_ok = (cu[0] == 0 && cu[num_reqs] == num_tokens) ? 1 : 0;
        s_base = make_int2(0, 0);
    }
    for (int i = tid; i < kTileBins; i += kPrepThreads) s_hist[i] = 0;
    __syncthreads();
    for (int r = tid; r < num_reqs; r += kPrepThreads)
        if (cu[r + 1] < cu[r]) s_ok = 0;
    __syncthreads();
    const bool all_ok = s_ok != 0;
    if (!all_ok && tid == 0) raise_error(err, kErrBadMeta);
    float w_units = 0.f;   // this thread's prefill work
    for (int round = 0; round < num_reqs; round += kPrepThreads) {
        const int r = round + tid;
        int2 n = make_int2(0, 0);   // x: decode blocks, y: prefill tiles
        int q = 0;
        if (r < num_reqs && all_ok) {
            q = cu[r + 1] - cu[r];
            const int c = ctx[r];
            const bool ok = c >= 0 && c <= max_context_len && q <= max_q_len &&
                            (long long)c + q <= (long long)max_blocks * kBlockSize;
            if (!ok) {
                if (q > 0) raise_error(err, kErrBadMeta);
            } else if (q == 1) {
                n.x = (c + 1 + kBlockSize - 1) / kBlockSize;
            } else if (q > 1) {
                n.y = (q + kPrefillTileTokens - 1) / kPrefillTileTokens;
                for (int t = 0; t < n.y; ++t) {
                    const int tok0 = t * kPrefillTileTokens, ntok = min(kPrefillTileTokens, q - tok0);
                    const int end = c + tok0 + ntok;   // keys of the tile's last row
                    const float u = (float)((end + 127) / 128) + kTileFixedUnits;
                    w_units += u;
                    atomicAdd(&s_hist[tile_bin(c, tok0, ntok)], 1);
                }
            }
        }
        const int2 incl = warp_incl_scan(n, lane);
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int2 wt = s_warp[lane];
            const int2 wi = warp_incl_scan(wt, lane);
            s_warp[lane] = make_int2(wi.x - wt.x, wi.y - wt.y);
        }
        __syncthreads();
        const int2 wex = s_warp[warp];
        const int2 base = s_base;
        const int dx = base.x + wex.x + incl.x - n.x;
        const int dz = base.y + wex.y + incl.y - n.y;
        (void)dz;
        if (r < num_reqs) {
            page_off[r] = dx;
        }
        __syncthreads();
        if (tid == kPrepThreads - 1) s_base = make_int2(dx + n.x, dz + n.y);
        __syncthreads();
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w_units += __shfl_xor_sync(0xffffffffu, w_units, o);
    if (lane == 0) s_w[warp] = w_units;
    // Prefill tile order: bins in decreasing key-tile count, each bin's tiles from its first
    // output slot on (exclusive scan of the counts from the top bin down; kTileBins ==
    // kPrepThreads, one bin per thread).
    const int2 tot = s_base;
    const bool emit = tot.y <= max_prefill_tiles;
    if (!emit && tid == 0) raise_error(err, kErrBadMeta);
    {
        const int bin = kTileBins - 1 - tid;
        const int cnt = s_hist[bin];
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        __syncthreads();
        if (lane == 31) s_warp[warp].x = incl;
        __syncthreads();
        if (warp == 0) {
            const int wt = s_warp[lane].x;
            int wi = wt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, wi, o);
                if (lane >= o) wi += u;
            }
            s_warp[lane].x = wi - wt;
        }
        __syncthreads();
        s_hist[bin] = s_warp[warp].x + incl - cnt;
        __syncthreads();
    }
    if (all_ok && emit) {
        for (int r = tid; r < num_reqs; r += kPrepThreads) {
            const int q = cu[r + 1] - cu[r];
            const int c = ctx[r];
            if (q < 2 || c < 0 || c > max_context_len || q > max_q_len ||
                (long long)c + q > (long long)max_blocks * kBlockSize)
                continue;
            const int nt = (q + kPrefillTileTokens - 1) / kPrefillTileTokens;
            for (int t = nt - 1; t >= 0; --t) {
                const int tok0 = t * kPrefillTileTokens, ntok = min(kPrefillTileTokens, q - tok0);
                const int at = atomicAdd(&s_hist[tile_bin(c, tok0, ntok)], 1);
                pre_tiles[at] = make_int4(r, tok0, ntok, 0);
            }
        }
    }
    __syncthreads();
    if (tid == 0) {
        float w = 0.f;
        for (int i = 0; i < kPrepThreads / 32; ++i) w += s_w[i];
        page_off[num_reqs] = tot.x;
        counters[1] = emit ? tot.y : 0;
        counters[2] = decode_sm_share(tot.x, w * kNumKvHeads, num_sms);
        counters[3] = 0;
        counters[4] = 0;
        counters[5] = 0;
        counters[6] = 0;
    }
    // This kernel reads nothing the previous one (kv_append) writes, so it ran alongside
    // it; it finishes only after that kernel has, so that later kernels, which wait for
    // this one, see the appended K/V.
    grid_dep_wait();
}

}  // namespace

StepLayout make_step_layout(int num_reqs, int num_tokens) {
    StepLayout L{};
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const int pre_reqs = num_reqs < num_tokens / 2 ? num_reqs : num_tokens / 2;
    L.max_prefill_tiles = num_tokens / kPrefillTileTokens + pre_reqs + 1;
    L.max_partials = num_reqs + kMaxDecodeCtas;
    size_t off = 0;
    L.counters_off = off;
    off = up(off + 8 * sizeof(int32_t));
    L.page_off_off = off;
    off = up(off + ((size_t)num_reqs + 1) * sizeof(int32_t));
    L.prefill_tiles_off = off;
    off = up(off + (size_t)L.max_prefill_tiles * sizeof(int4));
    L.part_acc_off = off;
    off = up(off + (size_t)L.max_partials * kNumQHeads * kHeadDim * sizeof(float));
    L.part_ml_off = off;
    off = up(off + (size_t)L.max_partials * kNumQHeads * sizeof(float2));
    L.total = off;
    return L;
}

cudaError_t launch_step_prep(const StepArgs& a, cudaStream_t stream) {
    const StepLayout& L = a.lay;
    return launch_pdl(step_prep_kernel, dim3(1), dim3(kPrepThreads), 0, stream, a.cu_seqlens_q, a.context_lens,
                      a.num_reqs, a.num_tokens, a.max_q_len, a.max_context_len, a.max_blocks_per_seq,
                      L.max_prefill_tiles, a.num_sms > 0 ? a.num_sms : 1,
                      reinterpret_cast<int32_t*>(a.ws + L.counters_off),
                      reinterpret_cast<int32_t*>(a.ws + L.page_off_off),
                      reinterpret_cast<int4*>(a.ws + L.prefill_tiles_off), a.err);
}

}  // namespace kvp
