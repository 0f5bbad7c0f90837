// Decode rows (q_len == 1): split-KV paged attention on CUDA cores, HBM-bound.
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
//   2,048 block ids a CTA stages).  A
//   CTA walks its range request by request; a request cut by a range boundary produces one
//   partial per CTA that touches it (slot r + cta), merged by whichever of those CTAs
//   finishes last; a request inside one range is finished in place.
// * The CTA first looks up the physical ids of all its blocks in parallel (into shared
//   memory), so no table lookup sits between a freed buffer and its refill.
// * One block of all 8 KV heads is 32 KiB contiguous in the pool, so each block of K and
//   of V arrives with ONE bulk copy (cp.async.bulk, mbarrier completion) into a 3-stage
//   ring of 64 KiB stages; the last of the 16 warps to finish with a stage refills it
//   with the block three ahead (no thread waits for the others to do so).
// * GQA packing: the 4 query heads of a KV head share every K/V byte read.  Two warps
//   per KV head (16 warps) split each block's 16 tokens 8/8, with separate
//   online-softmax states merged at the end of a request segment.
// * Scores: a lane holds 16 of the 128 dims (8 lanes per token) of 2 tokens for all 4
//   query heads; packed fp32x2 FMAs; a transpose-reduce over the 8 lanes (7 shuffles)
//   leaves one finished (token, head) score per lane.  Online softmax in base 2 (the
//   query is pre-scaled by softmax_scale * log2 e) against a reference max per head that
//   moves only when a score exceeds it by more than 2^8 (a warp vote; the max reduction
//   and the rescale run only then), with per-lane partial sums reduced once per segment.
// * P.V: a lane owns 4 output dims of all 4 heads; weights of the warp's 8 tokens go
//   through a per-warp shared-memory slot as duplicated pairs for the packed FMAs.
// Partial results keep (m, l, unnormalised acc); the last CTA to finish a split row
// (an arrival count per row) merges them: O = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M)
// l_s with M = max_s m_s.
// Keys at positions >= ctx + 1 of the last block are excluded (score -inf, value unread).
#include "kvp_device.cuh"
#include "kvp_launch.h"

namespace kvp {

namespace {

constexpr int kDecWarps = 16;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDecStages = 3;
constexpr int kTokensPerWarp = kBlockSize / 2;

constexpr int kIdCap = 2048;   // block ids a CTA stages in shared memory (its whole range)

struct __align__(128) DecodeSmem {
    uint8_t kv[kDecStages][2][kBlockBytes];           // [stage][K|V][8 heads x 16 x 128 bf16]
    int32_t ids[kIdCap];                              // physical block of each block of the range
    float2 pbuf[kDecWarps][kTokensPerWarp][kGroup];   // (p, p) per token and head
    float2 abuf[kDecWarps][kGroup];                   // (alpha, alpha) per head
    float2 merge_acc[kNumKvHeads][32][8];             // second half's accumulators
    float merge_ml[kNumKvHeads][8];                   // second half's m[4], l[4]
    int pair_abort[kNumKvHeads];
    int cta_abort;
    int merge_last;
    int first_req, last_req;
    unsigned released[kDecStages];                    // warps done with a stage (mod 16)
    int issued;                                       // blocks issued so far
    int n_rel;                                        // blocks in the range
    const uint8_t* cache[2];                          // K and V pools
    uint32_t* err;
    uint64_t policy;
    uint64_t full[kDecStages];
};

// atom.add with acquire-release ordering at CTA scope (shared memory).
__device__ __forceinline__ unsigned atomic_add_acq_rel_cta(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_u32(p)), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void named_bar(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) { return make_float2(bf16lo(w), bf16hi(w)); }

// Partial dot products of one token's 16-dim slice (chunks dg and dg + 8 of its 256-byte
// K row) with the 4 query heads' matching slices.
__device__ __forceinline__ void token_scores(const float2 (&q2)[kGroup][8], const uint8_t* krow, int dg,
                                             float (&v)[kGroup]) {
    const uint4 ka = *reinterpret_cast<const uint4*>(krow + dg * 16);
    const uint4 kb = *reinterpret_cast<const uint4*>(krow + 128 + dg * 16);
    const uint32_t w[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
    float2 s[kGroup];
#pragma unroll
    for (int g = 0; g < kGroup; ++g) s[g] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float2 k = bf16x2_to_f2(w[i]);
#pragma unroll
        for (int g = 0; g < kGroup; ++g) s[g] = __ffma2_rn(q2[g][i], k, s[g]);
    }
#pragma unroll
    for (int g = 0; g < kGroup; ++g) v[g] = s[g].x + s[g].y;
}

// acc[g] += p[g] * v for one token: v is the lane's 4 dims of the token's V row, p the
// token's weight for each of the 4 query heads (stored as duplicated pairs).
__device__ __forceinline__ void pv_token(const float2 (&pt)[kGroup], const uint8_t* vrow, int lane,
                                         float2 (&acc)[kGroup][2]) {
    const uint2 vv = *reinterpret_cast<const uint2*>(vrow + lane * 8);
    const float2 va = bf16x2_to_f2(vv.x), vb = bf16x2_to_f2(vv.y);
    const float4 p01 = *reinterpret_cast<const float4*>(&pt[0]);
    const float4 p23 = *reinterpret_cast<const float4*>(&pt[2]);
    const float2 pg[4] = {make_float2(p01.x, p01.y), make_float2(p01.z, p01.w), make_float2(p23.x, p23.y),
                          make_float2(p23.z, p23.w)};
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
        acc[g][0] = __ffma2_rn(va, pg[g], acc[g][0]);
        acc[g][1] = __ffma2_rn(vb, pg[g], acc[g][1]);
    }
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


// Copy K and V of block `q` of the range into stage `st`.
__device__ __noinline__ void issue_block(DecodeSmem& S, int st, int q) {
    const size_t off = (size_t)S.ids[q] * kBlockBytes;
    mbar_arrive_expect_tx(&S.full[st], 2 * kBlockBytes);
    bulk_load(S.kv[st][0], S.cache[0] + off, kBlockBytes, &S.full[st], S.policy);
    bulk_load(S.kv[st][1], S.cache[1] + off, kBlockBytes, &S.full[st], S.policy);
    atomicMax(&S.issued, q + 1);
}

// Lane 0 of a warp that is done reading block `rel` (stage st; the warp's reads are
// ordered before this by __syncwarp): the last of the 16 warps refills the stage with
// block rel + kDecStages.  One shared atomic per warp and block: the count both elects
// the refilling warp and orders every warp's reads (release) before the copy (acquire,
// then a proxy fence for the bulk copy's write).
__device__ __forceinline__ void release_stage(DecodeSmem& S, int st, int rel) {
    const unsigned old = atomic_add_acq_rel_cta(&S.released[st], 1u);
    if ((old & (kDecWarps - 1)) != kDecWarps - 1) return;
    const int q = rel + kDecStages;
    if (q >= S.n_rel) return;
    fence_proxy_async_smem();
    issue_block(S, st, q);
}

// Merge the partial results of a decode row whose blocks were split over CTAs c0..c1
// (all 512 threads of the CTA: thread t takes query head t / 16 and dims 8 (t % 16) ..
// 8 (t % 16) + 7).  O = sum_c 2^(m_c - M) acc_c / sum_c 2^(m_c - M) l_c.
__device__ __noinline__ void merge_partials(int r, int row, int c0, int c1, const float* part_acc,
                                            const float2* part_ml, __nv_bfloat16* out) {
    const int head = threadIdx.x >> 4, d0 = (threadIdx.x & 15) * 8;
    float M = -INFINITY;
    for (int c = c0; c <= c1; ++c) M = fmaxf(M, __ldcg(&part_ml[((size_t)r + c) * kNumQHeads + head]).x);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float L = 0.f, o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int c = c0; c <= c1; ++c) {
        const size_t sh = ((size_t)r + c) * kNumQHeads + head;
        const float2 ml = __ldcg(&part_ml[sh]);
        const float w = fast_exp2(ml.x - Mu);
        L = fmaf(ml.y, w, L);
        const float4 a = __ldcg(reinterpret_cast<const float4*>(part_acc + sh * kHeadDim + d0));
        const float4 b = __ldcg(reinterpret_cast<const float4*>(part_acc + sh * kHeadDim + d0 + 4));
        o[0] = fmaf(a.x, w, o[0]); o[1] = fmaf(a.y, w, o[1]); o[2] = fmaf(a.z, w, o[2]); o[3] = fmaf(a.w, w, o[3]);
        o[4] = fmaf(b.x, w, o[4]); o[5] = fmaf(b.y, w, o[5]); o[6] = fmaf(b.z, w, o[6]); o[7] = fmaf(b.w, w, o[7]);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint4 wv;
    wv.x = pack_bf16x2(o[0] * inv, o[1] * inv);
    wv.y = pack_bf16x2(o[2] * inv, o[3] * inv);
    wv.z = pack_bf16x2(o[4] * inv, o[5] * inv);
    wv.w = pack_bf16x2(o[6] * inv, o[7] * inv);
    *reinterpret_cast<uint4*>(out + (size_t)row * kQRowElems + head * kHeadDim + d0) = wv;
}

__global__ void __launch_bounds__(kDecThreads, 1) decode_kernel(
    const __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ out, const int32_t* __restrict__ cu,
    const int32_t* __restrict__ ctx, const int32_t* __restrict__ tables, int max_blocks, int num_blocks,
    const uint8_t* __restrict__ k_cache, const uint8_t* __restrict__ v_cache, const int32_t* __restrict__ page_off,
    int num_reqs, int wave, const int32_t* __restrict__ counters, float* __restrict__ part_acc,
    float2* __restrict__ part_ml,
    int32_t* __restrict__ seg_count, float scale_log2, uint32_t* __restrict__ err) {
    extern __shared__ uint8_t smem_raw[];
    DecodeSmem& S = *reinterpret_cast<DecodeSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
        S.cache[0] = k_cache;
        S.cache[1] = v_cache;
        S.err = err;
        S.policy = policy_evict_first();
        S.cta_abort = 0;
        fence_barrier_init();
    }
    if (threadIdx.x < kNumKvHeads) S.pair_abort[threadIdx.x] = 0;
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
        for (int j = 0; j < kDecStages && j < n_rel; ++j) issue_block(S, j, j);
    }

    const int h = warp >> 1, half = warp & 1;
    const int dg = lane & 7;                      // dims 8dg..8dg+7 and 64+8dg..64+8dg+7
    const int tl = lane >> 3;                     // token within a group of 4
    const int my_tok = (lane & 1) * 4 + tl;       // token (of the warp's 8) whose score this lane ends with
    const int hd = ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);  // ... and its head
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

        float2 q2[kGroup][8];
#pragma unroll
        for (int g = 0; g < kGroup; ++g) {
            const uint4* qp = reinterpret_cast<const uint4*>(q + (size_t)row * kQRowElems + (h * kGroup + g) * kHeadDim);
            const uint4 a = qp[dg], b = qp[8 + dg];
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 f = bf16x2_to_f2(w[i]);
                q2[g][i] = make_float2(f.x * scale_log2, f.y * scale_log2);
            }
        }
        float m_ref = -INFINITY, l_part = 0.f;   // per head hd (m_ref uniform over its lanes)
        float2 acc[kGroup][2];
#pragma unroll
        for (int g = 0; g < kGroup; ++g) acc[g][0] = acc[g][1] = make_float2(0.f, 0.f);

        for (; page < seg_end; ++page) {
            if (!aborted && !mbar_wait(&S.full[stage], phase)) {
                raise_error(err, kErrTimeout);
                aborted = true;
            }
            if (!aborted) {
                const uint8_t* kt = S.kv[stage][0] + h * kTileBytes + half * kTokensPerWarp * kHeadBytes;
                const int pos0 = (page - req_lo) * kBlockSize + half * kTokensPerWarp;
                const int n_valid = min(kTokensPerWarp, n_keys - pos0);   // >= 1 except in a last block
                // ---- scores of tokens tl and 4 + tl, all 4 heads
                const uint8_t* k0 = kt + tl * kHeadBytes;
                float v0[kGroup], v1[kGroup];
                token_scores(q2, k0, dg, v0);
                token_scores(q2, k0 + 4 * kHeadBytes, dg, v1);
                // transpose-reduce over the 8 lanes of a token: bit 2 picks the head pair,
                // bit 1 the head, bit 0 the token
                const bool b2 = (lane >> 2) & 1, b1 = (lane >> 1) & 1, b0 = lane & 1;
                float x[4], y[4];
                x[0] = b2 ? v0[2] : v0[0];
                x[1] = b2 ? v0[3] : v0[1];
                x[2] = b2 ? v1[2] : v1[0];
                x[3] = b2 ? v1[3] : v1[1];
                y[0] = b2 ? v0[0] : v0[2];
                y[1] = b2 ? v0[1] : v0[3];
                y[2] = b2 ? v1[0] : v1[2];
                y[3] = b2 ? v1[1] : v1[3];
#pragma unroll
                for (int k = 0; k < 4; ++k) x[k] += __shfl_xor_sync(0xffffffffu, y[k], 4);
                float u0 = b1 ? x[1] : x[0], u1 = b1 ? x[3] : x[2];
                const float t0 = b1 ? x[0] : x[1], t1 = b1 ? x[2] : x[3];
                u0 += __shfl_xor_sync(0xffffffffu, t0, 2);
                u1 += __shfl_xor_sync(0xffffffffu, t1, 2);
                float sc = b0 ? u1 : u0;
                sc += __shfl_xor_sync(0xffffffffu, b0 ? u0 : u1, 1);
                if (my_tok >= n_valid) sc = -INFINITY;
                // ---- online softmax for head hd over the warp's 8 tokens.  The reference
                // max m_ref moves only when a score exceeds it by more than 2^8 (then the
                // warp reduces the max and rescales); the sum stays a per-lane partial
                // until the segment ends.  Weights are 2^(s - m_ref) <= 2^8.
                if (__any_sync(0xffffffffu, sc > m_ref + 8.f)) {
                    float mx = sc;
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    const float m_new = fmaxf(m_ref, mx);
                    const float alpha = fast_exp2(m_ref - (m_new == -INFINITY ? 0.f : m_new));
                    l_part *= alpha;
                    m_ref = m_new;
                    if ((lane & 0x19) == 0) S.abuf[warp][hd] = make_float2(alpha, alpha);
                    __syncwarp();
                    const float4 al01 = *reinterpret_cast<const float4*>(&S.abuf[warp][0]);
                    const float4 al23 = *reinterpret_cast<const float4*>(&S.abuf[warp][2]);
                    const float2 al[4] = {make_float2(al01.x, al01.y), make_float2(al01.z, al01.w),
                                          make_float2(al23.x, al23.y), make_float2(al23.z, al23.w)};
#pragma unroll
                    for (int g = 0; g < kGroup; ++g) {
                        acc[g][0] = __fmul2_rn(acc[g][0], al[g]);
                        acc[g][1] = __fmul2_rn(acc[g][1], al[g]);
                    }
                }
                const float p = fast_exp2(sc - (m_ref == -INFINITY ? 0.f : m_ref));
                l_part += p;
                S.pbuf[warp][my_tok][hd] = make_float2(p, p);
                __syncwarp();
                {
                    const uint8_t* vt = S.kv[stage][1] + h * kTileBytes + half * kTokensPerWarp * kHeadBytes;
                    if (n_valid == kTokensPerWarp) {
#pragma unroll
                        for (int t = 0; t < kTokensPerWarp; ++t)
                            pv_token(S.pbuf[warp][t], vt + t * kHeadBytes, lane, acc);
                    } else {
                        for (int t = 0; t < n_valid; ++t) pv_token(S.pbuf[warp][t], vt + t * kHeadBytes, lane, acc);
                    }
                    __syncwarp();
                    if (lane == 0) release_stage(S, stage, page - lo);
                }
            }
            if (++stage == kDecStages) {
                stage = 0;
                phase ^= 1;
            }
        }

        // ------------------------------------------------ merge the two token halves
        l_part += __shfl_xor_sync(0xffffffffu, l_part, 1);
        l_part += __shfl_xor_sync(0xffffffffu, l_part, 8);
        l_part += __shfl_xor_sync(0xffffffffu, l_part, 16);
        float m[kGroup], l[kGroup];
#pragma unroll
        for (int g = 0; g < kGroup; ++g) {
            const int src = ((g >> 1) << 2) | ((g & 1) << 1);
            m[g] = __shfl_sync(0xffffffffu, m_ref, src);
            l[g] = __shfl_sync(0xffffffffu, l_part, src);
        }
        if (aborted && lane == 0) S.pair_abort[h] = 1;
        if (half == 1) {
#pragma unroll
            for (int g = 0; g < kGroup; ++g) {
                S.merge_acc[h][lane][2 * g] = acc[g][0];
                S.merge_acc[h][lane][2 * g + 1] = acc[g][1];
            }
            if (lane == 0) {
#pragma unroll
                for (int g = 0; g < kGroup; ++g) {
                    S.merge_ml[h][g] = m[g];
                    S.merge_ml[h][4 + g] = l[g];
                }
            }
        }
        named_bar(1 + h, 64);
        const bool pair_aborted = S.pair_abort[h] != 0;
        if (half == 0 && !pair_aborted) {
#pragma unroll
            for (int g = 0; g < kGroup; ++g) {
                const float m1 = S.merge_ml[h][g], l1 = S.merge_ml[h][4 + g];
                const float M = fmaxf(m[g], m1);
                const float Mu = (M == -INFINITY) ? 0.f : M;
                const float e0 = fast_exp2(m[g] - Mu), e1 = fast_exp2(m1 - Mu);
                const float L = l[g] * e0 + l1 * e1;
                const float2 b0 = S.merge_acc[h][lane][2 * g], b1 = S.merge_acc[h][lane][2 * g + 1];
                const float o0 = acc[g][0].x * e0 + b0.x * e1, o1 = acc[g][0].y * e0 + b0.y * e1;
                const float o2 = acc[g][1].x * e0 + b1.x * e1, o3 = acc[g][1].y * e0 + b1.y * e1;
                const int head = h * kGroup + g;
                if (whole) {
                    const float inv = L > 0.f ? 1.f / L : 0.f;
                    uint2 wv;
                    wv.x = pack_bf16x2(o0 * inv, o1 * inv);
                    wv.y = pack_bf16x2(o2 * inv, o3 * inv);
                    *reinterpret_cast<uint2*>(out + (size_t)row * kQRowElems + head * kHeadDim + lane * 4) = wv;
                } else {
                    const size_t slot = (size_t)r + blockIdx.x;
                    *reinterpret_cast<float4*>(part_acc + (slot * kNumQHeads + head) * kHeadDim + lane * 4) =
                        make_float4(o0, o1, o2, o3);
                    if (lane == 0) part_ml[slot * kNumQHeads + head] = make_float2(M, L);
                }
            }
        }
        named_bar(1 + h, 64);
        // The whole CTA agrees on abort before anyone leaves the loop (every warp walks the
        // same segments, so every warp reaches these barriers).
        if (pair_aborted && (warp & 1) == 0 && lane == 0) S.cta_abort = 1;
        __syncthreads();
        const bool cta_aborted = S.cta_abort != 0;
        if (!whole && !cta_aborted) {
            // Split row: count this CTA's partial in; the CTA that completes the count
            // merges all of the row's partials (their writes are published by the fence
            // before the count, and read past L1 after it).
            if (threadIdx.x == 0) {
                __threadfence();
                const int c0 = owner_cta(req_lo, P, G), c1 = owner_cta(req_hi - 1, P, G);
                const int old = atomicAdd(&seg_count[r], 1);
                S.merge_last = (old == c1 - c0) ? 1 : 0;
                if (S.merge_last) __threadfence();
            }
            __syncthreads();
            if (S.merge_last) merge_partials(r, row, owner_cta(req_lo, P, G), owner_cta(req_hi - 1, P, G), part_acc,
                                             part_ml, out);
            __syncthreads();
        }
        if (cta_aborted) break;
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

cudaError_t launch_decode(const StepArgs& a, cudaStream_t stream) {
    const StepLayout& L = a.lay;
    const size_t smem = sizeof(DecodeSmem) + 128;
    const int wave = decode_wave(a);
    return launch_pdl(decode_kernel, dim3(decode_grid(a, wave)), dim3(kDecThreads), smem, stream,
                      static_cast<const __nv_bfloat16*>(a.q), static_cast<__nv_bfloat16*>(a.out), a.cu_seqlens_q,
                      a.context_lens, a.block_tables, a.max_blocks_per_seq, a.num_blocks,
                      static_cast<const uint8_t*>(a.k_cache), static_cast<const uint8_t*>(a.v_cache),
                      reinterpret_cast<const int32_t*>(a.ws + L.page_off_off), a.num_reqs, wave,
                      reinterpret_cast<const int32_t*>(a.ws + L.counters_off),
                      reinterpret_cast<float*>(a.ws + L.part_acc_off), reinterpret_cast<float2*>(a.ws + L.part_ml_off),
                      reinterpret_cast<int32_t*>(a.ws + L.seg_count_off), a.softmax_scale * 1.4426950408889634f, a.err);
}

cudaError_t configure_decode_kernel() {
    return cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(sizeof(DecodeSmem) + 128));
}

}  // namespace kvp
