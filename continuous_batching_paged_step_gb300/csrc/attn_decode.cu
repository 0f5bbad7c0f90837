// Decode rows (q_len == 1): split-KV paged attention on CUDA cores, HBM-bound.
//
// The decode formula of page "Continuous Batching" (k4i.top), section "与 KV cache 的关
// 系": the row's query attends to [K_cache; k_t] and [V_cache; v_t] of its own request,
// i.e. all positions 0 .. ctx of that request (this step's key was appended already).
// Decode streams the whole KV history every step (same page, section "为什么 decode 是
// bandwidth-bound"), so the kernel is built to keep HBM busy:
//
// * Work item = (request, chunk of up to `chunk_pages` 16-token blocks).  One block of
//   all 8 KV heads is 32 KiB contiguous in the pool, so each block of K and of V arrives
//   with ONE bulk copy (cp.async.bulk, mbarrier completion) into a 3-stage shared-memory
//   ring: 64 KiB per stage, 192 KiB in flight per SM.  A dedicated producer warp runs
//   ahead across pages and items; the kernel is persistent (one CTA per SM, items taken
//   round-robin).
// * GQA packing: the 4 query heads of a KV head share every K/V byte read.  Two consumer
//   warps per KV head (16 warps) split each block's 16 tokens 8/8 and keep separate
//   online-softmax states, merged at the end of the item.
// * Scores: a lane holds 16 of the 128 dims of one token (8 lanes per token, 4 tokens per
//   pass) for all 4 query heads; a 3-step transpose-reduce over the 8 lanes (4 shuffles)
//   leaves one finished score per lane.  Online softmax in base 2 (scores pre-scaled by
//   softmax_scale * log2 e) with running max m and sum l per head.
// * P.V: a lane owns 4 output dims of all 4 heads; weights come from a per-warp
//   shared-memory slot (broadcast reads); fp32 accumulation.
// * A request with one chunk writes its bf16 output directly; otherwise each chunk writes
//   (m, l, unnormalised acc) to the workspace and the combine kernel merges them:
//   O = sum_c 2^(m_c - M) acc_c / sum_c 2^(m_c - M) l_c.
// Keys at positions >= ctx + 1 in the last block are excluded (score -inf, value unread).
#include "kvp_device.cuh"
#include "kvp_launch.h"

namespace kvp {

namespace {

constexpr int kDecConsumerWarps = 16;
constexpr int kDecThreads = (kDecConsumerWarps + 1) * 32;
constexpr int kDecStages = 3;
constexpr int kTokensPerWarp = kBlockSize / 2;

struct __align__(128) DecodeSmem {
    uint8_t kv[kDecStages][2][kBlockBytes];                 // [stage][K|V][8 heads x 16 x 128 bf16]
    float4 pbuf[kDecConsumerWarps][kTokensPerWarp];          // softmax weights of 4 heads per token
    float4 abuf[kDecConsumerWarps];                          // rescale factors of 4 heads
    float merge_acc[kNumKvHeads][32][16];                    // second half's accumulators
    float merge_ml[kNumKvHeads][8];                          // second half's m[4], l[4]
    int pair_abort[kNumKvHeads];
    uint64_t full[kDecStages];
    uint64_t empty[kDecStages];
};

__device__ __forceinline__ void named_bar(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
    f[0] = bf16lo(u.x); f[1] = bf16hi(u.x);
    f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
    f[4] = bf16lo(u.z); f[5] = bf16hi(u.z);
    f[6] = bf16lo(u.w); f[7] = bf16hi(u.w);
}

__global__ void __launch_bounds__(kDecThreads, 1) decode_kernel(
    const __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ out, const int32_t* __restrict__ cu,
    const int32_t* __restrict__ ctx, const int32_t* __restrict__ tables, int max_blocks, int num_blocks,
    const uint8_t* __restrict__ k_cache, const uint8_t* __restrict__ v_cache, const int32_t* __restrict__ counters,
    const int4* __restrict__ items, float* __restrict__ part_acc, float2* __restrict__ part_ml, float scale_log2,
    uint32_t* __restrict__ err) {
    extern __shared__ uint8_t smem_raw[];
    DecodeSmem& S = *reinterpret_cast<DecodeSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_items = counters[0];
    if ((int)blockIdx.x >= n_items) return;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kDecStages; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], kDecConsumerWarps);
        }
        fence_barrier_init();
    }
    if (threadIdx.x < kNumKvHeads) S.pair_abort[threadIdx.x] = 0;
    __syncthreads();

    if (warp == kDecConsumerWarps) {
        // ---------------------------------------------------------------- producer
        if (lane != 0) return;
        const uint64_t pol = policy_evict_first();
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            const int4 item = items[it];
            const int32_t* trow = tables + (size_t)item.x * max_blocks + item.y;
            for (int j = 0; j < item.z; ++j) {
                int b = trow[j];
                if ((unsigned)b >= (unsigned)num_blocks) {
                    raise_error(err, kErrBadBlock);
                    b = 0;
                }
                if (!mbar_wait(&S.empty[stage], phase ^ 1)) {
                    raise_error(err, kErrTimeout);
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&S.full[stage], 2 * kBlockBytes);
                bulk_load(S.kv[stage][0], k_cache + (size_t)b * kBlockBytes, kBlockBytes, &S.full[stage], pol);
                bulk_load(S.kv[stage][1], v_cache + (size_t)b * kBlockBytes, kBlockBytes, &S.full[stage], pol);
                ++issued;
                if (++stage == kDecStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        // Drain: the CTA must not retire while a copy still targets its shared memory.
        for (int k = 1; k <= kDecStages && k <= issued; ++k) {
            int s = stage - k;
            uint32_t ph = phase;
            if (s < 0) {
                s += kDecStages;
                ph ^= 1;
            }
            if (!mbar_wait(&S.full[s], ph)) raise_error(err, kErrTimeout);
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    const int h = warp >> 1, half = warp & 1;
    const int dg = lane & 7;                 // 16-dim slice: dims 8dg..8dg+7 and 64+8dg..64+8dg+7
    const int tl = lane >> 3;                // token within a pass of 4
    const int hd = ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);  // head whose score this lane ends with
    int stage = 0;
    uint32_t phase = 0;
    bool aborted = false;

    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const int4 item = items[it];
        const int r = item.x, first_page = item.y, npages = item.z, slot = item.w;
        const int row = cu[r];
        const int n_keys = ctx[r] + 1;

        float qf[kGroup][16];
#pragma unroll
        for (int g = 0; g < kGroup; ++g) {
            const uint4* qp = reinterpret_cast<const uint4*>(q + (size_t)row * kQRowElems + (h * kGroup + g) * kHeadDim);
            float t[8];
            bf16x8_to_f32(qp[dg], t);
#pragma unroll
            for (int i = 0; i < 8; ++i) qf[g][i] = t[i] * scale_log2;
            bf16x8_to_f32(qp[8 + dg], t);
#pragma unroll
            for (int i = 0; i < 8; ++i) qf[g][8 + i] = t[i] * scale_log2;
        }
        float m_own = -INFINITY, l_own = 0.f;
        float acc[kGroup][4];
#pragma unroll
        for (int g = 0; g < kGroup; ++g)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[g][i] = 0.f;

        for (int j = 0; j < npages; ++j) {
            if (!aborted && !mbar_wait(&S.full[stage], phase)) {
                raise_error(err, kErrTimeout);
                aborted = true;
            }
            if (!aborted) {
                const uint8_t* kt = S.kv[stage][0] + h * kTileBytes;
                const uint8_t* vt = S.kv[stage][1] + h * kTileBytes;
                const int pos0 = (first_page + j) * kBlockSize;
                float sc[2];
#pragma unroll
                for (int a = 0; a < 2; ++a) {
                    const int tok = half * kTokensPerWarp + a * 4 + tl;
                    const uint4 k0 = *reinterpret_cast<const uint4*>(kt + tok * kHeadBytes + dg * 16);
                    const uint4 k1 = *reinterpret_cast<const uint4*>(kt + tok * kHeadBytes + 128 + dg * 16);
                    float kf[16];
                    bf16x8_to_f32(k0, kf);
                    bf16x8_to_f32(k1, kf + 8);
                    float v[kGroup];
#pragma unroll
                    for (int g = 0; g < kGroup; ++g) {
                        float s = 0.f;
#pragma unroll
                        for (int i = 0; i < 16; ++i) s = fmaf(qf[g][i], kf[i], s);
                        v[g] = s;
                    }
                    // transpose-reduce over the 8 lanes of this token
                    const bool b2 = (lane >> 2) & 1;
                    float k_lo = b2 ? v[2] : v[0], k_hi = b2 ? v[3] : v[1];
                    const float s_lo = b2 ? v[0] : v[2], s_hi = b2 ? v[1] : v[3];
                    k_lo += __shfl_xor_sync(0xffffffffu, s_lo, 4);
                    k_hi += __shfl_xor_sync(0xffffffffu, s_hi, 4);
                    const bool b1 = (lane >> 1) & 1;
                    float kk = b1 ? k_hi : k_lo;
                    kk += __shfl_xor_sync(0xffffffffu, b1 ? k_lo : k_hi, 2);
                    kk += __shfl_xor_sync(0xffffffffu, kk, 1);
                    sc[a] = (pos0 + tok < n_keys) ? kk : -INFINITY;
                }
                float mx = fmaxf(sc[0], sc[1]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float m_new = fmaxf(m_own, mx);
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                const float alpha = fast_exp2(m_own - m_use);
                const float p0 = fast_exp2(sc[0] - m_use), p1 = fast_exp2(sc[1] - m_use);
                float ps = p0 + p1;
                ps += __shfl_xor_sync(0xffffffffu, ps, 8);
                ps += __shfl_xor_sync(0xffffffffu, ps, 16);
                l_own = l_own * alpha + ps;
                m_own = m_new;
                float* pw = reinterpret_cast<float*>(&S.pbuf[warp][0]);
                if ((lane & 1) == 0) {
                    pw[tl * 4 + hd] = p0;
                    pw[(4 + tl) * 4 + hd] = p1;
                }
                if ((lane & 0x19) == 0) reinterpret_cast<float*>(&S.abuf[warp])[hd] = alpha;
                __syncwarp();
                const float4 al = S.abuf[warp];
                const float alv[4] = {al.x, al.y, al.z, al.w};
#pragma unroll
                for (int g = 0; g < kGroup; ++g)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[g][i] *= alv[g];
#pragma unroll
                for (int t = 0; t < kTokensPerWarp; ++t) {
                    const int tok = half * kTokensPerWarp + t;
                    if (pos0 + tok < n_keys) {
                        const uint2 vv = *reinterpret_cast<const uint2*>(vt + tok * kHeadBytes + lane * 8);
                        const float v0 = bf16lo(vv.x), v1 = bf16hi(vv.x), v2 = bf16lo(vv.y), v3 = bf16hi(vv.y);
                        const float4 pp = S.pbuf[warp][t];
                        const float pg[4] = {pp.x, pp.y, pp.z, pp.w};
#pragma unroll
                        for (int g = 0; g < kGroup; ++g) {
                            acc[g][0] = fmaf(pg[g], v0, acc[g][0]);
                            acc[g][1] = fmaf(pg[g], v1, acc[g][1]);
                            acc[g][2] = fmaf(pg[g], v2, acc[g][2]);
                            acc[g][3] = fmaf(pg[g], v3, acc[g][3]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.empty[stage]);
            }
            if (++stage == kDecStages) {
                stage = 0;
                phase ^= 1;
            }
        }

        // ------------------------------------------------ merge the two token halves
        float m[kGroup], l[kGroup];
#pragma unroll
        for (int g = 0; g < kGroup; ++g) {
            const int src = ((g >> 1) << 2) | ((g & 1) << 1);
            m[g] = __shfl_sync(0xffffffffu, m_own, src);
            l[g] = __shfl_sync(0xffffffffu, l_own, src);
        }
        if (aborted && lane == 0) S.pair_abort[h] = 1;
        if (half == 1) {
#pragma unroll
            for (int g = 0; g < kGroup; ++g)
#pragma unroll
                for (int i = 0; i < 4; ++i) S.merge_acc[h][lane][g * 4 + i] = acc[g][i];
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
                float o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) o[i] = acc[g][i] * e0 + S.merge_acc[h][lane][g * 4 + i] * e1;
                const int head = h * kGroup + g;
                if (slot < 0) {
                    const float inv = L > 0.f ? 1.f / L : 0.f;
                    uint2 w;
                    w.x = pack_bf16x2(o[0] * inv, o[1] * inv);
                    w.y = pack_bf16x2(o[2] * inv, o[3] * inv);
                    *reinterpret_cast<uint2*>(out + (size_t)row * kQRowElems + head * kHeadDim + lane * 4) = w;
                } else {
                    *reinterpret_cast<float4*>(part_acc + ((size_t)slot * kNumQHeads + head) * kHeadDim + lane * 4) =
                        make_float4(o[0], o[1], o[2], o[3]);
                    if (lane == 0) part_ml[(size_t)slot * kNumQHeads + head] = make_float2(M, L);
                }
            }
        }
        named_bar(1 + h, 64);
        if (pair_aborted) break;
    }
}

// Merge the split-KV partials of one decode row: one warp per (request, query head),
// a lane owns 4 output dims.
__global__ void __launch_bounds__(256) combine_kernel(const int32_t* __restrict__ counters,
                                                      const int4* __restrict__ combines,
                                                      const int32_t* __restrict__ cu,
                                                      const float* __restrict__ part_acc,
                                                      const float2* __restrict__ part_ml,
                                                      __nv_bfloat16* __restrict__ out) {
    const int e = blockIdx.x;
    if (e >= counters[2]) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int head = blockIdx.y * 8 + warp;
    const int4 c = combines[e];
    const int row = cu[c.x];
    float M = -INFINITY;
    for (int k = 0; k < c.z; ++k) M = fmaxf(M, part_ml[(size_t)(c.y + k) * kNumQHeads + head].x);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float L = 0.f, o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
    for (int k = 0; k < c.z; ++k) {
        const size_t sh = (size_t)(c.y + k) * kNumQHeads + head;
        const float2 ml = part_ml[sh];
        const float w = fast_exp2(ml.x - Mu);
        L = fmaf(ml.y, w, L);
        const float4 a = *reinterpret_cast<const float4*>(part_acc + sh * kHeadDim + lane * 4);
        o0 = fmaf(a.x, w, o0);
        o1 = fmaf(a.y, w, o1);
        o2 = fmaf(a.z, w, o2);
        o3 = fmaf(a.w, w, o3);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint2 wv;
    wv.x = pack_bf16x2(o0 * inv, o1 * inv);
    wv.y = pack_bf16x2(o2 * inv, o3 * inv);
    *reinterpret_cast<uint2*>(out + (size_t)row * kQRowElems + head * kHeadDim + lane * 4) = wv;
}

}  // namespace

cudaError_t launch_decode(const StepArgs& a, cudaStream_t stream) {
    const StepLayout& L = a.lay;
    if (L.max_decode_items <= 0) return cudaSuccess;
    int grid = a.num_sms;
    if (grid > L.max_decode_items) grid = L.max_decode_items;
    const size_t smem = sizeof(DecodeSmem) + 128;
    decode_kernel<<<grid, kDecThreads, smem, stream>>>(
        static_cast<const __nv_bfloat16*>(a.q), static_cast<__nv_bfloat16*>(a.out), a.cu_seqlens_q, a.context_lens,
        a.block_tables, a.max_blocks_per_seq, a.num_blocks, static_cast<const uint8_t*>(a.k_cache),
        static_cast<const uint8_t*>(a.v_cache), reinterpret_cast<const int32_t*>(a.ws + L.counters_off),
        reinterpret_cast<const int4*>(a.ws + L.decode_items_off), reinterpret_cast<float*>(a.ws + L.part_acc_off),
        reinterpret_cast<float2*>(a.ws + L.part_ml_off), a.softmax_scale * 1.4426950408889634f, a.err);
    return cudaGetLastError();
}

cudaError_t launch_combine(const StepArgs& a, cudaStream_t stream) {
    const StepLayout& L = a.lay;
    if (L.max_combines <= 0) return cudaSuccess;
    dim3 grid(L.max_combines, kNumQHeads / 8);
    combine_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const int32_t*>(a.ws + L.counters_off),
                                             reinterpret_cast<const int4*>(a.ws + L.combines_off), a.cu_seqlens_q,
                                             reinterpret_cast<const float*>(a.ws + L.part_acc_off),
                                             reinterpret_cast<const float2*>(a.ws + L.part_ml_off),
                                             static_cast<__nv_bfloat16*>(a.out));
    return cudaGetLastError();
}

cudaError_t configure_decode_kernel() {
    return cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(sizeof(DecodeSmem) + 128));
}

}  // namespace kvp
