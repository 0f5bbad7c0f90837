// Prefill-chunk rows (q_len >= 2): paged attention on the 5th-generation tensor cores.
//
// A prefill chunk attends to the KV that earlier chunks left in the cache plus its own
// rows, causally (page "Continuous Batching 深入实现", section "第三层：Chunked Prefill";
// page "11.2 连续批处理与 PagedAttention", section 11.2.2, Figure 11-3: per head the
// scores are Q[q, 128] x K^T[128, ctx + q] with a causal mask).  These are dense
// contractions, so they run as tcgen05.mma (bf16 operands in shared memory, fp32
// accumulators in TMEM).
//
// CTA = one (request, 32-token q tile, KV head g).  The 128 MMA rows are the 32 tokens x
// the 4 query heads that share KV head g (row = 4 * token + head), so every K/V tile is
// loaded once for the whole GQA group.  Key tiles are 128 keys = 8 blocks of 16: each
// block's (block, head g) 4 KiB tile is fetched by two 2-D TMA loads (one per 64-dim
// half, 128-byte swizzle), landing in the canonical K-major SW128 layout.
//
// Warp roles (8 warps): warp 0 lane 0 issues TMA loads (Q once, then K/V tiles into a
// 2-stage ring); warp 1 owns TMEM (512 columns: S double buffer at 0 and 128, O at 256)
// and lane 0 issues the MMAs; warps 4-7 run the softmax, one thread per MMA row (TMEM
// lane), and the epilogue.  Per key tile kt:
//   MMA   : S[kt%2] = Q K_kt^T            (issued one tile ahead)
//   soft  : m_new = max(m, rowmax S * scale * log2 e); P = 2^(S' - m_new) as bf16;
//           l = l * 2^(m - m_new) + sum P; once O is stable (previous P V done) rescale O
//           in TMEM by 2^(m - m_new) when it changed; write P to shared memory
//           (K-major SW128)
//   MMA   : O += P V_kt                   (V read MN-major: keys are the K dimension)
// End: O / l rounded to bf16 and stored for the tile's valid rows.
// Masking: key position > row position gets -inf (only on tiles that reach past the
// tile's first row position); V rows at positions >= ctx + q_len in the last tile are
// zeroed in shared memory so stale bytes cannot leak into P V.
#include <cuda.h>

#include "kvp_device.cuh"
#include "kvp_launch.h"

namespace kvp {

namespace {

constexpr int kPreThreads = 256;
constexpr int kKeyTile = 128;
constexpr int kHalfBytes = 16384;   // 128 rows x 128 bytes (64 bf16)

struct __align__(1024) PrefillSmem {
    uint8_t q[2][kHalfBytes];        // [d half][128 rows]
    uint8_t k[2][2][kHalfBytes];     // [stage][d half][128 keys]
    uint8_t v[2][2][kHalfBytes];     // [stage][d half][128 keys]
    uint8_t p[2][kHalfBytes];        // [key half][128 rows]
    uint64_t q_full;
    uint64_t k_full[2], v_full[2], kv_empty[2];
    uint64_t s_full[2], s_free[2];
    uint64_t p_full, o_ready, mma_done;
    uint32_t tmem_base;
};

struct PrefillArgs {
    const int32_t* counters;
    const int4* tiles;
    const int32_t* cu;
    const int32_t* ctx;
    const int32_t* tables;
    int max_blocks;
    int num_blocks;
    __nv_bfloat16* out;
    uint32_t* err;
    float scale_log2;
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

__global__ void __launch_bounds__(kPreThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    PrefillSmem& S =
        *reinterpret_cast<PrefillSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tile = blockIdx.x, g = blockIdx.y;
    if (tile >= a.counters[1]) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int4 td = a.tiles[tile];
    const int r = td.x, tok0 = td.y, ntok = td.z;
    const int ctx_r = a.ctx[r];
    const int q_len = a.cu[r + 1] - a.cu[r];
    const int row0 = a.cu[r] + tok0;
    const int qpos0 = ctx_r + tok0;
    const int qpos_last = qpos0 + ntok - 1;
    const int n_keys = ctx_r + q_len;
    const int n_pages = (n_keys + kBlockSize - 1) / kBlockSize;
    const int n_kt = qpos_last / kKeyTile + 1;

    if (warp == 1) {
        tmem_alloc(&S.tmem_base, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        mbar_init(&S.q_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&S.k_full[s], 1);
            mbar_init(&S.v_full[s], 1);
            mbar_init(&S.kv_empty[s], 1);
            mbar_init(&S.s_full[s], 1);
            mbar_init(&S.s_free[s], 4);
        }
        mbar_init(&S.p_full, 4);
        mbar_init(&S.o_ready, 1);
        mbar_init(&S.mma_done, 1);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            prefetch_tmap(&tmap_q);
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
            mbar_arrive_expect_tx(&S.q_full, 2 * kHalfBytes);
            tma_load_3d(S.q[0], &tmap_q, 0, g * kGroup, row0, &S.q_full);
            tma_load_3d(S.q[1], &tmap_q, 64, g * kGroup, row0, &S.q_full);
            const int32_t* trow = a.tables + (size_t)r * a.max_blocks;
            int issued = 0;
            for (int kt = 0; kt < n_kt; ++kt) {
                const int s = kt & 1;
                if (!mbar_wait(&S.kv_empty[s], ((kt >> 1) & 1) ^ 1)) {
                    raise_error(a.err, kErrTimeout);
                    break;
                }
                const int pg0 = kt * (kKeyTile / kBlockSize);
                const int npg = min(kKeyTile / kBlockSize, n_pages - pg0);
                int rows[kKeyTile / kBlockSize];
#pragma unroll
                for (int j = 0; j < kKeyTile / kBlockSize; ++j) {
                    int b = j < npg ? trow[pg0 + j] : 0;
                    if ((unsigned)b >= (unsigned)a.num_blocks) {
                        raise_error(a.err, kErrBadBlock);
                        b = 0;
                    }
                    rows[j] = (b * kNumKvHeads + g) * kBlockSize;
                }
                mbar_arrive_expect_tx(&S.k_full[s], npg * kTileBytes);
                for (int j = 0; j < npg; ++j) {
                    tma_load_2d(S.k[s][0] + j * 2048, &tmap_k, 0, rows[j], &S.k_full[s]);
                    tma_load_2d(S.k[s][1] + j * 2048, &tmap_k, 64, rows[j], &S.k_full[s]);
                }
                mbar_arrive_expect_tx(&S.v_full[s], npg * kTileBytes);
                for (int j = 0; j < npg; ++j) {
                    tma_load_2d(S.v[s][0] + j * 2048, &tmap_v, 0, rows[j], &S.v_full[s]);
                    tma_load_2d(S.v[s][1] + j * 2048, &tmap_v, 64, rows[j], &S.v_full[s]);
                }
                ++issued;
            }
            // Drain: wait until every copy issued into this CTA's shared memory landed.
            if (!mbar_wait(&S.q_full, 0)) raise_error(a.err, kErrTimeout);
            for (int kt = issued - 2 < 0 ? 0 : issued - 2; kt < issued; ++kt) {
                const int s = kt & 1;
                const uint32_t ph = (kt >> 1) & 1;
                if (!mbar_wait(&S.k_full[s], ph) || !mbar_wait(&S.v_full[s], ph)) raise_error(a.err, kErrTimeout);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, 0);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, 1);
            const uint32_t sq = smem_u32(S.q[0]), sp = smem_u32(S.p[0]);
            bool ok = mbar_wait(&S.q_full, 0);
            auto issue_qk = [&](int j) -> bool {
                const int s = j & 1;
                if (!mbar_wait(&S.k_full[s], (j >> 1) & 1)) return false;
                if (j >= 2 && !mbar_wait(&S.s_free[s], ((j >> 1) - 1) & 1)) return false;
                tc_fence_after();
                const uint32_t sk = smem_u32(S.k[s][0]);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t koff = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                    tc_mma_f16(tmem + s * 128, smem_desc_sw128(sq + koff, 16, 1024),
                               smem_desc_sw128(sk + koff, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
                }
                tc_commit(&S.s_full[s]);
                return true;
            };
            if (ok) ok = issue_qk(0);
            for (int kt = 0; kt < n_kt && ok; ++kt) {
                if (kt + 1 < n_kt && !(ok = issue_qk(kt + 1))) break;
                const int s = kt & 1;
                if (!mbar_wait(&S.p_full, kt & 1) || !mbar_wait(&S.v_full[s], (kt >> 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sv = smem_u32(S.v[s][0]);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t poff = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                    tc_mma_f16(tmem + 256, smem_desc_sw128(sp + poff, 16, 1024),
                               smem_desc_sw128(sv + kk * 2048, kHalfBytes, 1024), idesc_pv,
                               (kt > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&S.o_ready);
                tc_commit(&S.kv_empty[s]);
            }
            if (!ok) raise_error(a.err, kErrTimeout);
            // No MMA may still be running when TMEM is released.
            tc_commit(&S.mma_done);
            if (!mbar_wait(&S.mma_done, 0)) raise_error(a.err, kErrTimeout);
        }
    } else if (warp >= 4) {
        // --------------------------------------------------------- softmax + epilogue
        const int wq = warp - 4;
        const int row = wq * 32 + lane;
        const int tl = row >> 2, hl = row & 3;
        const bool row_valid = tl < ntok;
        const int qpos = row_valid ? qpos0 + tl : -1;
        const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int kt = 0; kt < n_kt; ++kt) {
            const int s = kt & 1;
            if (!warp_wait(&S.s_full[s], (kt >> 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) tmem_ld32(t_lane + s * 128 + cc * 32, sr[cc]);
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.s_free[s]);

            const int key0 = kt * kKeyTile;
            const bool need_mask = key0 + kKeyTile - 1 > qpos0;
            float mx = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float f = __uint_as_float(sr[cc][i]) * a.scale_log2;
                    if (need_mask && key0 + cc * 32 + i > qpos) f = -INFINITY;
                    sr[cc][i] = __float_as_uint(f);
                    mx = fmaxf(mx, f);
                }
            const float m_new = fmaxf(m, mx);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = fast_exp2(m - m_use);
            float sum = 0.f;
            uint32_t pk[64];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float p0 = fast_exp2(__uint_as_float(sr[cc][i]) - m_use);
                    const float p1 = fast_exp2(__uint_as_float(sr[cc][i + 1]) - m_use);
                    sum += p0 + p1;
                    pk[cc * 16 + i / 2] = pack_bf16x2(p0, p1);
                }
            l = l * alpha + sum;
            m = m_new;

            if (kt > 0) {
                // O is stable once the previous P V has completed; P's buffer is free too.
                if (!warp_wait(&S.o_ready, (kt - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(t_lane + 256 + cc * 32, o);
                        tc_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(t_lane + 256 + cc * 32, o);
                    }
                    tc_wait_st();
                }
            }
            if (kt == n_kt - 1 && key0 + kKeyTile > n_keys) {
                // keys at positions >= n_keys hold stale bytes: zero their V rows
                if (!warp_wait(&S.v_full[s], (kt >> 1) & 1)) {
                    ok = false;
                    break;
                }
                if (key0 + row >= n_keys) {
                    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        *reinterpret_cast<uint4*>(S.v[s][0] + row * 128 + c * 16) = z;
                        *reinterpret_cast<uint4*>(S.v[s][1] + row * 128 + c * 16) = z;
                    }
                }
            }
            // P row -> shared memory, K-major with 128-byte swizzle (16-byte chunk c of
            // row r sits at chunk position c ^ (r % 8) within the row's 128 bytes).
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint4 w = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                *reinterpret_cast<uint4*>(S.p[c >> 3] + row * 128 + (((c & 7) ^ (row & 7)) << 4)) = w;
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.p_full);
        }
        if (ok && warp_wait(&S.o_ready, (n_kt - 1) & 1)) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16* orow = a.out + (size_t)(row0 + tl) * kQRowElems + (g * kGroup + hl) * kHeadDim;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t o[32];
                tmem_ld32(t_lane + 256 + cc * 32, o);
                tc_wait_ld();
                if (row_valid) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(o[8 * c + 0]) * inv, __uint_as_float(o[8 * c + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(o[8 * c + 2]) * inv, __uint_as_float(o[8 * c + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(o[8 * c + 4]) * inv, __uint_as_float(o[8 * c + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(o[8 * c + 6]) * inv, __uint_as_float(o[8 * c + 7]) * inv);
                        *reinterpret_cast<uint4*>(orow + cc * 32 + c * 8) = w;
                    }
                }
            }
        } else {
            raise_error(a.err, kErrTimeout);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_prefill(const StepArgs& a, const CUtensorMap* tmap_q, const CUtensorMap* tmap_k,
                           const CUtensorMap* tmap_v, cudaStream_t stream) {
    const StepLayout& L = a.lay;
    if (L.max_prefill_tiles <= 0 || a.max_q_len < 2) return cudaSuccess;
    PrefillArgs pa;
    pa.counters = reinterpret_cast<const int32_t*>(a.ws + L.counters_off);
    pa.tiles = reinterpret_cast<const int4*>(a.ws + L.prefill_tiles_off);
    pa.cu = a.cu_seqlens_q;
    pa.ctx = a.context_lens;
    pa.tables = a.block_tables;
    pa.max_blocks = a.max_blocks_per_seq;
    pa.num_blocks = a.num_blocks;
    pa.out = static_cast<__nv_bfloat16*>(a.out);
    pa.err = a.err;
    pa.scale_log2 = a.softmax_scale * 1.4426950408889634f;
    dim3 grid(L.max_prefill_tiles, kNumKvHeads);
    const size_t smem = sizeof(PrefillSmem) + 1024;
    prefill_kernel<<<grid, kPreThreads, smem, stream>>>(*tmap_q, *tmap_k, *tmap_v, pa);
    return cudaGetLastError();
}

cudaError_t configure_prefill_kernel() {
    return cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(sizeof(PrefillSmem) + 1024));
}

}  // namespace kvp
