// Decode rows (q_len == 1): split-KV paged attention, HBM-bound.
//
// The decode formula of page "Continuous Batching" (k4i.top), section "与 KV cache 的关
// 系": the row's query attends to [K_cache; k_t] and [V_cache; v_t] of its own request,
// i.e. all positions 0 .. ctx of that request (this step's key was appended already).
// Decode streams the whole KV history every step (same page, section "为什么 decode 是
// bandwidth-bound"), so the kernel is built to keep HBM busy:
//
// * Balanced split: the 16-token blocks of all decode rows, concatenated in request
//   order (page_off[r] = first global block of request r), are cut into equal contiguous
//   ranges, one per CTA (one CTA per SM of the decode's share of the SMs, which the step's
//   metadata kernel sizes so that the prefill tiles run on the others; fewer CTAs when
//   there are under 4 blocks per CTA; more, in whole waves, when a range would exceed the
//   2,048 block ids a CTA stages).  A CTA walks its range request by request; a request
//   cut by a range boundary produces one partial per CTA that touches it (slot r + cta),
//   merged by whichever of those CTAs finishes last; a request inside one range is
//   finished in place.
// * The CTA first looks up the physical ids of all its blocks in parallel (into shared
//   memory), so no table lookup sits between a freed buffer and its refill.
// * One block of all 8 KV heads is 128 rows (head x token) of 128 dims in the pool, so
//   its K and its V arrive with four tensor-map loads (one per 64-dim half, 128-byte
//   swizzle) into a 3-stage ring of 64 KiB stages; the last of the 8 warps to finish
//   with a stage refills it with the block three ahead (no thread waits for the others
//   to do so).
// * One warp per KV head.  Its 4 query heads share every K/V byte (GQA packing), and the
//   two contractions of a block are small matrix products, which run on the tensor
//   cores (mma.sync m16n8k16, bf16 operands, fp32 accumulation) instead of as thousands
//   of scalar FMAs:  S^T = K Q^T (16 tokens x 8 columns, the 4 query heads and 4 zero
//   columns) and O^T += V^T P^T (128 dims x 8 columns).  K and V fragments come from
//   the swizzled tiles with ldmatrix (V transposed on the way), so reads are free of
//   bank conflicts; the weights go from the score fragment to the P^T operand with one
//   register transpose (movmatrix) per 8 tokens.
// * Online softmax in base 2 (scores x softmax_scale x log2 e) against a reference max
//   per head that moves only when a score exceeds it by more than 2^8 (a warp vote; the
//   max reduction and the rescale run only then), with per-lane partial sums reduced
//   once per request segment.  Weights enter P.V rounded to bf16; the sums use them
//   unrounded.
// Partial results keep (m, l, unnormalised acc); the last CTA to finish a split row
// (an arrival count per row) merges them: O = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M)
// l_s with M = max_s m_s.
// A warp reads all of its K and V fragments of a block into registers before anything
// else and releases the stage at once, so a stage is held only for those reads.
// Keys at positions >= ctx + 1 of the last block are excluded: score -inf, and their V
// values zeroed in the fragments (stale bytes could hold NaN, and 0 x NaN is NaN).
#include <cuda.h>

#include "kvp_device.cuh"
#include "kvp_launch.h"

namespace kvp {

namespace {

constexpr int kDecWarps = kNumKvHeads;   // one warp per KV head
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDecStages = 3;
constexpr int kBlockRows = kNumKvHeads * kBlockSize;   // rows (head, token) of one block: 128
constexpr int kHalfTile = kBlockRows * 128;            // one block's 64-dim half: 128 rows x 128 B
constexpr int kStageBytes = 4 * kHalfTile;             // K and V, two halves each: 64 KiB

constexpr int kIdCap = 2048;   // block ids a CTA stages in shared memory (its whole range)

struct __align__(1024) DecodeSmem {
    uint8_t kv[kDecStages][2][2][kHalfTile];   // [stage][K|V][dim half][row 16 h + token], 128-byte swizzle
    int32_t ids[kIdCap];                       // physical block of each block of the range
    int cta_abort;
    int merge_last;
    int first_req, last_req;
    unsigned released[kDecStages];             // warps done with a stage (mod 8)
    int issued;                                // blocks issued so far
    int n_rel;                                 // blocks in the range
    uint64_t policy;
    uint64_t full[kDecStages];
};

// Tensor-map load with an L2 eviction hint.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* tmap, int c0, int c1, uint32_t bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(tmap), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
        : "memory");
}

// Four 8x8 bf16 matrices from shared memory (lanes 8j..8j+7 give the row addresses of
// matrix j); .trans delivers each matrix transposed.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// d += A (16x16, row-major fragments) x B (16x8, column fragments), bf16 in, fp32 out.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 bf16 matrix held one row pair per lane (lane 4i + j holds row i,
// columns 2j and 2j + 1).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Copy K and V of block `q` of the range into stage `st`.
__device__ __forceinline__ void issue_block(DecodeSmem& S, const CUtensorMap* tk, const CUtensorMap* tv, int st,
                                            int q) {
    const int y = S.ids[q] * kBlockRows;
    const uint32_t bar = smem_u32(&S.full[st]);
    const uint32_t d = smem_u32(S.kv[st][0][0]);
    mbar_arrive_expect_tx(&S.full[st], kStageBytes);
    tma_load_2d_hint(d, tk, 0, y, bar, S.policy);
    tma_load_2d_hint(d + kHalfTile, tk, 64, y, bar, S.policy);
    tma_load_2d_hint(d + 2 * kHalfTile, tv, 0, y, bar, S.policy);
    tma_load_2d_hint(d + 3 * kHalfTile, tv, 64, y, bar, S.policy);
    atomicMax(&S.issued, q + 1);
}

// atom.add with acquire-release ordering at CTA scope (shared memory).
__device__ __forceinline__ unsigned atomic_add_acq_rel_cta(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_u32(p)), "r"(v) : "memory");
    return old;
}

// Lane 0 of a warp that is done reading block `rel` (stage st; the warp's reads are
// ordered before this by __syncwarp): the last of the 8 warps refills the stage with
// block rel + kDecStages.  One shared atomic per warp and block: the count both elects
// the refilling warp and orders every warp's accesses (release) before the copy
// (acquire, then a proxy fence for the tensor copy's write).
__device__ __forceinline__ void release_stage(DecodeSmem& S, const CUtensorMap* tk, const CUtensorMap* tv, int st,
                                              int rel) {
    const unsigned old = atomic_add_acq_rel_cta(&S.released[st], 1u);
    if ((old & (kDecWarps - 1)) != kDecWarps - 1) return;
    const int q = rel + kDecStages;
    if (q >= S.n_rel) return;
    fence_proxy_async_smem();
    issue_block(S, tk, tv, st, q);
}

// A decode CTA streams at least this many blocks: with fewer blocks than CTAs x this,
// only ceil(P / kMinBlocksPerCta) CTAs take part (fewer, longer segments to merge).
constexpr int kMinBlocksPerCta = 4;

// CTAs that share P blocks: at most `wave` at a time (one per SM), each range at most
// kIdCap blocks (whole extra waves when P needs them).  0 when the launch is too small.
__device__ __forceinline__ int decode_ctas_used(int P, int wave, int grid) {
    const int per_wave = max(1, min(wave, (P + kMinBlocksPerCta - 1) / kMinBlocksPerCta));
    const long long waves = max(1LL, ((long long)P + (long long)per_wave * kIdCap - 1) / ((long long)per_wave * kIdCap));
    const long long G = waves * per_wave;
    return G > grid ? 0 : (int)G;
}

// Block range [lo, hi) of CTA c out of G over P blocks.
__device__ __forceinline__ void cta_range(int P, int c, int G, int& lo, int& hi) {
    lo = (int)(((long long)P * c) / G);
    hi = (int)(((long long)P * (c + 1)) / G);
}

// The CTA whose range holds global block x.
__device__ __forceinline__ int owner_cta(int x, int P, int G) {
    return (int)((((long long)x + 1) * G - 1) / P);
}


// Merge the partial results of a decode row whose blocks were split over CTAs c0..c1
// (all 256 threads of the CTA: thread t takes query head t / 8 and dims 16 (t % 8) ..
// 16 (t % 8) + 15).  O = sum_c 2^(m_c - M) acc_c / sum_c 2^(m_c - M) l_c.
__device__ __noinline__ void merge_partials(int r, int row, int c0, int c1, const float* part_acc,
                                            const float2* part_ml, __nv_bfloat16* out) {
    const int head = threadIdx.x >> 3, d0 = (threadIdx.x & 7) * 16;
    float M = -INFINITY;
    for (int c = c0; c <= c1; ++c) M = fmaxf(M, __ldcg(&part_ml[((size_t)r + c) * kNumQHeads + head]).x);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float L = 0.f, o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i] = 0.f;
    for (int c = c0; c <= c1; ++c) {
        const size_t sh = ((size_t)r + c) * kNumQHeads + head;
        const float2 ml = __ldcg(&part_ml[sh]);
        const float w = fast_exp2(ml.x - Mu);
        L = fmaf(ml.y, w, L);
        const float4* src = reinterpret_cast<const float4*>(part_acc + sh * kHeadDim + d0);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 a = __ldcg(src + j);
            o[4 * j + 0] = fmaf(a.x, w, o[4 * j + 0]);
            o[4 * j + 1] = fmaf(a.y, w, o[4 * j + 1]);
            o[4 * j + 2] = fmaf(a.z, w, o[4 * j + 2]);
            o[4 * j + 3] = fmaf(a.w, w, o[4 * j + 3]);
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint4* dst = reinterpret_cast<uint4*>(out + (size_t)row * kQRowElems + head * kHeadDim + d0);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        uint4 wv;
        wv.x = pack_bf16x2(o[8 * j + 0] * inv, o[8 * j + 1] * inv);
        wv.y = pack_bf16x2(o[8 * j + 2] * inv, o[8 * j + 3] * inv);
        wv.z = pack_bf16x2(o[8 * j + 4] * inv, o[8 * j + 5] * inv);
        wv.w = pack_bf16x2(o[8 * j + 6] * inv, o[8 * j + 7] * inv);
        dst[j] = wv;
    }
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

__global__ void __launch_bounds__(kDecThreads, 1) decode_kernel(
    const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
    const __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ out, const int32_t* __restrict__ cu,
    const int32_t* __restrict__ ctx, const int32_t* __restrict__ tables, int max_blocks, int num_blocks,
    const int32_t* __restrict__ page_off, int num_reqs, int wave, const int32_t* __restrict__ counters,
    float* __restrict__ part_acc, float2* __restrict__ part_ml, int32_t* __restrict__ seg_count, float scale_log2,
    uint32_t* __restrict__ err) {
    extern __shared__ uint8_t smem_raw[];
    DecodeSmem& S =
        *reinterpret_cast<DecodeSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    grid_dep_wait();     // block offsets, cache contents
    grid_dep_launch();
    const int P = page_off[num_reqs];
    if (P <= 0) return;
    // SMs left to this step's prefill tiles run them meanwhile (unless the launch is too
    // small for the narrower waves that would need)
    int G = decode_ctas_used(P, max(1, min(wave, counters[2])), gridDim.x);
    if (G == 0) G = decode_ctas_used(P, wave, gridDim.x);
    if (G == 0) {
        // the launch has too few CTAs for this many blocks (the host sizes it from an
        // upper bound, so this means inconsistent metadata)
        if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(err, kErrBadMeta);
        return;
    }
    if ((int)blockIdx.x >= G) return;
    int lo, hi;
    cta_range(P, blockIdx.x, G, lo, hi);
    if (lo >= hi) return;
    const int n_rel = hi - lo;   // <= kIdCap by construction of G
    if (n_rel > kIdCap) {
        if (threadIdx.x == 0) raise_error(err, kErrBadMeta);
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kDecStages; ++s) {
            mbar_init(&S.full[s], 1);
            S.released[s] = 0;
        }
        S.issued = 0;
        S.n_rel = n_rel;
        S.policy = policy_evict_first();
        S.cta_abort = 0;
        fence_barrier_init();
    }
    // requests holding the first and the last block of the range (one parallel pass)
    for (int r = threadIdx.x; r < num_reqs; r += kDecThreads) {
        const int a0 = page_off[r], a1 = page_off[r + 1];
        if (a0 <= lo && lo < a1) S.first_req = r;
        if (a0 <= hi - 1 && hi - 1 < a1) S.last_req = r;
    }
    __syncthreads();
    // physical id of every block of the range
    {
        const int r_first = S.first_req, r_last = S.last_req;
        for (int x = lo + threadIdx.x; x < hi; x += kDecThreads) {
            int ra = r_first, rb = r_last;   // largest r with page_off[r] <= x
            while (ra < rb) {
                const int mid = (ra + rb + 1) >> 1;
                if (page_off[mid] <= x) ra = mid;
                else rb = mid - 1;
            }
            int b = tables[(size_t)ra * max_blocks + (x - page_off[ra])];
            if ((unsigned)b >= (unsigned)num_blocks) {
                raise_error(err, kErrBadBlock);
                b = 0;
            }
            S.ids[x - lo] = b;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int j = 0; j < kDecStages && j < n_rel; ++j) issue_block(S, &tmap_k, &tmap_v, j, j);

    }

    // Fragment coordinates (PTX mma.m16n8k16 layouts): lane = 4 g + t.  A fragment rows
    // are tokens (S^T) or dims (O^T); B columns and C columns are the query heads, of
    // which columns 0..3 are real (lanes with t < 2 hold them in C).
    const int h = warp;
    const int g = lane >> 2, t = lane & 3;
    const int x7 = lane & 7;
    // ldmatrix row addresses inside a stage's K (V) region, 64-dim half 0: K row = token
    // x7 + 8 (lane bit 3), 16-byte chunk 2j + (lane bit 4) of the k-step's 32 bytes; V row
    // = token x7 + 8 (lane bit 4), chunk 2j + (lane bit 3); 128-byte swizzle: chunk ^ row % 8.
    uint32_t k_off[4], v_off[4];
    {
        const uint32_t k_row = (uint32_t)(h * kBlockSize + x7 + 8 * ((lane >> 3) & 1)) * 128;
        const uint32_t v_row = (uint32_t)(h * kBlockSize + x7 + 8 * (lane >> 4)) * 128;
        const uint32_t k_cb = lane >> 4, v_cb = (lane >> 3) & 1;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            k_off[j] = k_row + ((((uint32_t)(2 * j) + k_cb) ^ (uint32_t)x7) << 4);
            v_off[j] = v_row + ((((uint32_t)(2 * j) + v_cb) ^ (uint32_t)x7) << 4);
        }
    }
    const uint32_t ring0 = smem_u32(S.kv[0][0][0]);
    int stage = 0;
    uint32_t phase = 0;
    bool aborted = false;

    int r = S.first_req;
    int page = lo;
    while (page < hi) {
        const int req_lo = page_off[r], req_hi = page_off[r + 1];
        const int seg_end = min(hi, req_hi);
        const bool whole = (page == req_lo) && (seg_end == req_hi);
        const int row = cu[r];
        const int n_keys = ctx[r] + 1;

        // Q^T as the B operand of S^T = K Q^T: k-step s covers dims 16 s .. 16 s + 15; lane
        // (g, t) holds head g's dims 16 s + 2 t, +1 and 16 s + 2 t + 8, +9 (zero for g >= 4)
        uint32_t qb[8][2];
        {
            const uint32_t* qw = reinterpret_cast<const uint32_t*>(q + (size_t)row * kQRowElems +
                                                                    (h * kGroup + (g & 3)) * kHeadDim);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                qb[s][0] = g < kGroup ? __ldg(qw + 8 * s + t) : 0u;
                qb[s][1] = g < kGroup ? __ldg(qw + 8 * s + 4 + t) : 0u;
            }
        }
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // heads 2t, 2t + 1
        float o[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

        for (; page < seg_end; ++page) {
            if (!aborted && *reinterpret_cast<volatile int*>(&S.cta_abort)) aborted = true;   // another warp gave up
            if (!aborted && !warp_wait(&S.full[stage], phase)) {
                if (lane == 0) {
                    raise_error(err, kErrTimeout);
                    S.cta_abort = 1;
                }
                aborted = true;
            }
            if (!aborted) {
                const uint32_t kb = ring0 + stage * kStageBytes, vb = kb + 2 * kHalfTile;
                const int n_valid = n_keys - (page - req_lo) * kBlockSize;   // >= 1; < 16 only in a last block
                // All of this warp's reads of the stage first (K and V fragments into
                // registers), then the stage is released, so the refill starts before the
                // arithmetic rather than after it.
                uint32_t ka[8][4], va[8][4];
#pragma unroll
                for (int s = 0; s < 8; ++s) ldsm_x4(kb + (s >> 2) * kHalfTile + k_off[s & 3], ka[s]);
#pragma unroll
                for (int i = 0; i < 8; ++i) ldsm_x4_t(vb + (i >> 2) * kHalfTile + v_off[i & 3], va[i]);
                __syncwarp();
                if (lane == 0) release_stage(S, &tmap_k, &tmap_v, stage, page - lo);
                if (n_valid < kBlockSize) {
                    // tokens past the end of the request: zero their V values (stale bytes
                    // could hold NaN, and 0 x NaN is NaN).  V^T fragment registers 0, 1 hold
                    // tokens 2t, 2t + 1; registers 2, 3 tokens 2t + 8, 2t + 9.
                    auto keep = [&](int tk) -> uint32_t {
                        return (tk < n_valid ? 0x0000FFFFu : 0u) | (tk + 1 < n_valid ? 0xFFFF0000u : 0u);
                    };
                    const uint32_t k01 = keep(2 * t), k89 = keep(2 * t + 8);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        va[i][0] &= k01;
                        va[i][1] &= k01;
                        va[i][2] &= k89;
                        va[i][3] &= k89;
                    }
                }
                // ---- S^T = K Q^T: 16 tokens x (4 heads + 4 zero columns)
                float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int s = 0; s < 8; s += 2) {
                    mma_16816(sa, ka[s], qb[s][0], qb[s][1]);
                    mma_16816(sb, ka[s + 1], qb[s + 1][0], qb[s + 1][1]);
                }
                // lane holds tokens g, g + 8 of heads 2t, 2t + 1: x[0] (g, 2t), x[1] (g, 2t+1),
                // x[2] (g+8, 2t), x[3] (g+8, 2t+1)
                float x[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) x[j] = (sa[j] + sb[j]) * scale_log2;
                if (t >= 2 || g >= n_valid) x[0] = x[1] = -INFINITY;
                if (t >= 2 || g + 8 >= n_valid) x[2] = x[3] = -INFINITY;
                // ---- online softmax against the lazily moved reference max
                const bool need = fmaxf(x[0], x[2]) > m0 + 8.f || fmaxf(x[1], x[3]) > m1 + 8.f;
                if (__any_sync(0xffffffffu, need)) {
                    float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                    }
                    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
                    const float a0 = fast_exp2(m0 - (n0 == -INFINITY ? 0.f : n0));
                    const float a1 = fast_exp2(m1 - (n1 == -INFINITY ? 0.f : n1));
                    l0 *= a0;
                    l1 *= a1;
                    m0 = n0;
                    m1 = n1;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        o[i][0] *= a0;
                        o[i][1] *= a1;
                        o[i][2] *= a0;
                        o[i][3] *= a1;
                    }
                }
                const float u0 = m0 == -INFINITY ? 0.f : m0, u1 = m1 == -INFINITY ? 0.f : m1;
                const float p0 = fast_exp2(x[0] - u0), p1 = fast_exp2(x[1] - u1);
                const float p2 = fast_exp2(x[2] - u0), p3 = fast_exp2(x[3] - u1);
                l0 += p0 + p2;
                l1 += p1 + p3;
                // P^T as the B operand: lane (g, t) gets head g's weights of tokens 2t, 2t+1
                // (first 8 tokens) and 2t + 8, 2t + 9 (last 8)
                const uint32_t pb0 = movmatrix_t(pack_bf16x2(p0, p1));
                const uint32_t pb1 = movmatrix_t(pack_bf16x2(p2, p3));
                // ---- O^T += V^T P^T: m-tile i covers dims 16 i .. 16 i + 15
#pragma unroll
                for (int i = 0; i < 8; ++i) mma_16816(o[i], va[i], pb0, pb1);
            }
            if (++stage == kDecStages) {
                stage = 0;
                phase ^= 1;
            }
        }

        // ------------------------------------------------ finish the segment
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        if (!aborted) {
            if (whole) {
                // O = O^T / l, transposed back so that lane (g, t) holds dims 16 i + 2t, +1
                // and 16 i + 8 + 2t, +1 of head g
                const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
                uint32_t* orow = reinterpret_cast<uint32_t*>(out + (size_t)row * kQRowElems +
                                                             (h * kGroup + (g & 3)) * kHeadDim);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t w0 = movmatrix_t(pack_bf16x2(o[i][0] * i0, o[i][1] * i1));
                    const uint32_t w1 = movmatrix_t(pack_bf16x2(o[i][2] * i0, o[i][3] * i1));
                    if (g < kGroup) {
                        orow[8 * i + t] = w0;
                        orow[8 * i + 4 + t] = w1;
                    }
                }
            } else if (t < 2) {
                const size_t slot = (size_t)r + blockIdx.x;
                float* pa = part_acc + (slot * kNumQHeads + h * kGroup + 2 * t) * kHeadDim;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    pa[16 * i + g] = o[i][0];
                    pa[kHeadDim + 16 * i + g] = o[i][1];
                    pa[16 * i + 8 + g] = o[i][2];
                    pa[kHeadDim + 16 * i + 8 + g] = o[i][3];
                }
                if (g == 0) {
                    part_ml[slot * kNumQHeads + h * kGroup + 2 * t] = make_float2(m0, l0);
                    part_ml[slot * kNumQHeads + h * kGroup + 2 * t + 1] = make_float2(m1, l1);
                }
            }
        }
        if (!whole) {
            // Split row: once every warp's partial is written, count this CTA's partial
            // in; the CTA that completes the count merges all of the row's partials
            // (their writes are published by the fence before the count, and read past
            // L1 after it).  Every warp walks the same segments (an aborted warp skips
            // only the work), so every warp reaches these barriers.
            __syncthreads();
            const bool cta_aborted = S.cta_abort != 0;
            if (!cta_aborted && threadIdx.x == 0) {
                __threadfence();
                const int c0 = owner_cta(req_lo, P, G), c1 = owner_cta(req_hi - 1, P, G);
                const int old = atomicAdd(&seg_count[r], 1);
                S.merge_last = (old == c1 - c0) ? 1 : 0;
                if (S.merge_last) __threadfence();
            }
            __syncthreads();
            if (!cta_aborted && S.merge_last)
                merge_partials(r, row, owner_cta(req_lo, P, G), owner_cta(req_hi - 1, P, G), part_acc, part_ml, out);
            __syncthreads();
        }
        // next request that has blocks
        ++r;
        while (r + 1 <= num_reqs - 1 && page_off[r + 1] == page_off[r]) ++r;
    }

    // Drain: the CTA must not retire while a copy still targets its shared memory (only
    // possible after a wait ran out; otherwise every issued block was consumed).
    __syncthreads();
    if (threadIdx.x == 0) {
        const int n = S.issued;
        for (int j = max(0, n - kDecStages); j < n; ++j)
            if (!mbar_wait(&S.full[j % kDecStages], (uint32_t)((j / kDecStages) & 1))) raise_error(err, kErrTimeout);
    }
}

// CTAs that run at once: one per SM, or fewer when the pool asks for fewer.
int decode_wave(const StepArgs& a) {
    int w = a.num_sms > 0 ? a.num_sms : 1;
    if (w > kMaxDecodeCtas) w = kMaxDecodeCtas;
    if (a.decode_ctas > 0 && a.decode_ctas < w) w = a.decode_ctas;
    return w;
}

// Launch size: whole waves, enough that no CTA's share exceeds kIdCap blocks for the
// largest decode work these arguments allow (every request a decode row at the maximum
// context); capped at kMaxDecodeCtas (the kernel flags a step that would need more).
int decode_grid(const StepArgs& a, int wave) {
    const long long per_req = ((long long)a.max_context_len + 1 + kBlockSize - 1) / kBlockSize;
    const long long p_upper = per_req * (long long)a.num_reqs;
    const long long per_launch_wave = (long long)wave * kIdCap;
    long long waves = (p_upper + per_launch_wave - 1) / per_launch_wave;
    if (waves < 1) waves = 1;
    const long long max_waves = kMaxDecodeCtas / wave;
    if (waves > max_waves) waves = max_waves > 0 ? max_waves : 1;
    return (int)(waves * wave);
}

}  // namespace

cudaError_t launch_decode(const StepArgs& a, const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                          cudaStream_t stream) {
    const StepLayout& L = a.lay;
    const size_t smem = sizeof(DecodeSmem) + 1024;
    const int wave = decode_wave(a);
    return launch_pdl(decode_kernel, dim3(decode_grid(a, wave)), dim3(kDecThreads), smem, stream, *tmap_k, *tmap_v,
                      static_cast<const __nv_bfloat16*>(a.q), static_cast<__nv_bfloat16*>(a.out), a.cu_seqlens_q,
                      a.context_lens, a.block_tables, a.max_blocks_per_seq, a.num_blocks,
                      reinterpret_cast<const int32_t*>(a.ws + L.page_off_off), a.num_reqs, wave,
                      reinterpret_cast<const int32_t*>(a.ws + L.counters_off),
                      reinterpret_cast<float*>(a.ws + L.part_acc_off), reinterpret_cast<float2*>(a.ws + L.part_ml_off),
                      reinterpret_cast<int32_t*>(a.ws + L.seg_count_off), a.softmax_scale * 1.4426950408889634f, a.err);
}

cudaError_t configure_decode_kernel() {
    return cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(sizeof(DecodeSmem) + 1024));
}

}  // namespace kvp
