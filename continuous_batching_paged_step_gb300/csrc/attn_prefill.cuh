// Device code of the prefill chunks' tcgen05 attention, shared by the prefill kernel and
// the mixed step kernel (included by attn_prefill.cu and attn_mixed.cu).
//
// Prefill-chunk rows (q_len >= 2): paged attention on the 5th-generation tensor cores.
//
// A prefill chunk attends to the KV that earlier chunks left in the cache plus its own
// rows, causally (page "Continuous Batching 深入实现", section "第三层：Chunked Prefill";
// page "11.2 连续批处理与 PagedAttention", section 11.2.2, Figure 11-3: per head the
// scores are Q[q, 128] x K^T[128, ctx + q] with a causal mask).  These are dense
// contractions, so they run as tcgen05.mma (bf16 operands, fp32 accumulators in TMEM).
//
// CTA = one (request, 64-token q tile, KV head g), split into two MMA tiles A and B of
// 32 tokens each.  The 128 rows of an MMA tile are its 32 tokens x the 4 query heads that
// share KV head g (row = 4 * token + head), so every K/V tile is loaded once for the
// whole GQA group and serves both MMA tiles.  Key tiles are 128 keys = 8 blocks of 16:
// each block's (block, head g) 4 KiB tile is fetched by two 2-D TMA loads (one per 64-dim
// half, 128-byte swizzle), landing in the canonical K-major SW128 layout.
//
// Warp roles (12 warps): warp 0 issues the TMA loads of Q (once) and of K tiles into a
// 3-stage ring, warp 2 those of V tiles into a 2-stage ring; warp 1 owns TMEM and issues
// the MMAs (the warp in step, one elected lane issuing); warps 4-7 run the softmax of
// tile A and warps 8-11 that of tile B, one thread per MMA row (TMEM lane).  TMEM (512
// columns): one S buffer shared by the two tiles at 0, P of A at 128 and of B at 192 (bf16
// pairs, 64 columns each), O of A at 256 and of B at 384.  With P in columns of its own,
// S is free again as soon as a softmax has loaded it into registers, so the next Q K^T
// need not wait for the P V of the same tile: per key tile kt the MMA warp issues
// S = Q_A K_kt^T, then (once the softmax of A has read S) S = Q_B K_kt^T, then the P V of
// both tiles for key tile kt - 1.  A tile's softmax then runs beside three groups of MMAs
// (the other tile's Q K^T and both P V) instead of one.  Per key tile a softmax thread:
// reads its whole S row from TMEM in one load and frees S,
// keeps a running max m in base 2 (scores x softmax_scale x log2 e) that moves only when
// the tile's max exceeds it by more than 8 (then O and l are rescaled in place, after the
// tile's previous P V has completed: until then weights stay below 2^8, which bf16 and
// fp32 hold exactly enough), writes P = 2^(s - m) as bf16 pairs into its P columns (once
// the previous P V has read them), and the P V MMA reads P from TMEM as its A operand (V
// from shared memory, MN-major: keys are the K dimension).
// End: O / l rounded to bf16 for the tile's valid rows.
// Masking: key position > row position gets weight 0 (only on key tiles that reach past
// the tile's first row position); V rows at positions >= ctx + q_len in the last key
// tile are zeroed in shared memory so stale bytes cannot leak into P V.
#pragma once

#include <cuda.h>

#include "kvp_device.cuh"
#include "kvp_launch.h"

namespace kvp {

namespace {

constexpr int kPreThreads = 384;
constexpr int kKeyTile = 128;
constexpr int kHalfBytes = 16384;   // 128 rows x 128 bytes (64 bf16)
constexpr int kMmaTokens = kPrefillMmaTokens;   // tokens of one MMA tile (x 4 heads = 128 rows)
constexpr float kRescaleThreshold = 8.f;
// K is needed one softmax earlier than V, so its ring is deeper: 3 K + 2 V stages of
// 32 KiB, with Q (64 KiB) 224 KiB of shared memory.
constexpr int kKStages = 3;
constexpr int kVStages = 2;

static_assert(kPrefillTileTokens == 2 * kMmaTokens, "a CTA tile is two MMA tiles");

struct __align__(1024) PrefillSmem {
    uint8_t q[2][2][kHalfBytes];     // [MMA tile][d half][128 rows]
    uint8_t k[kKStages][2][kHalfBytes];   // [stage][d half][128 keys]
    uint8_t v[kVStages][2][kHalfBytes];   // [stage][d half][128 keys]
    uint64_t q_full;
    uint64_t k_full[kKStages], k_empty[kKStages];
    uint64_t v_full[kVStages], v_empty[kVStages];
    uint64_t s_full[2], p_full[2], pv_done[2];   // per MMA tile
    uint64_t s_free[2];   // tile t's softmax (4 warps) has read the shared S buffer
    uint64_t mma_done;
    uint32_t tmem_base;
};

struct PrefillArgs {
    const int32_t* counters;
    int32_t* done;               // CTAs that have finished (zeroed by the metadata kernel)
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

// Softmax and epilogue of one MMA tile (a warpgroup, one thread per row).
__device__ __forceinline__ void softmax_tile(PrefillSmem& S, const PrefillArgs& a, uint32_t tmem, int t, int wq,
                                             int lane, int g, int row0, int qpos0, int ntok_t, int nt, int n_kt,
                                             int n_keys, bool zero_v_rows) {
    const int row = wq * 32 + lane;
    const int tl = row >> 2, hl = row & 3;
    const bool row_valid = tl < ntok_t;
    const int tq0 = qpos0 + kMmaTokens * t;          // position of the tile's first token
    const int qpos = row_valid ? tq0 + tl : -1;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off;
    const uint32_t t_p = tmem + 128 + t * 64 + lane_off;
    const uint32_t t_o = tmem + 256 + t * 128 + lane_off;
    const float sc = a.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int kt = 0; kt < nt; ++kt) {
        if (!warp_wait(&S.s_full[t], kt & 1)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const int key0 = kt * kKeyTile;
        const bool need_mask = key0 + kKeyTile - 1 > tq0;
        // the whole S row in one TMEM load; then S is free for the next Q K^T
        uint32_t sr[128];
        tmem_ld128(t_s, sr);
        tc_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.s_free[t]);
        // O and the P columns are this tile's previous P V's until it has completed
        bool pv_clear = kt == 0;
        if (need_mask) {
            const int lim = qpos - key0;   // column i is visible iff i <= lim
#pragma unroll
            for (int i = 0; i < 128; ++i)
                if (i > lim) sr[i] = __float_as_uint(-INFINITY);
        }
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < 128; i += 8) {
            mx[0] = fmax3(mx[0], __uint_as_float(sr[i]), __uint_as_float(sr[i + 1]));
            mx[1] = fmax3(mx[1], __uint_as_float(sr[i + 2]), __uint_as_float(sr[i + 3]));
            mx[2] = fmax3(mx[2], __uint_as_float(sr[i + 4]), __uint_as_float(sr[i + 5]));
            mx[3] = fmax3(mx[3], __uint_as_float(sr[i + 6]), __uint_as_float(sr[i + 7]));
        }
        const float mx_s = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sc;
        const bool need = mx_s > m_used + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
            const float m_new = fmaxf(m_used, mx_s);
            const float alpha = (m_used == -INFINITY) ? 0.f : fast_exp2(m_used - m_new);
            if (kt > 0) {
                if (!warp_wait(&S.pv_done[t], (kt - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                pv_clear = true;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[32];
                    tmem_ld32(t_o + c * 32, o);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(t_o + c * 32, o);
                }
                tc_wait_st();
            }
            l *= alpha;
            m_used = m_new;
        }
        const float m_sub = (m_used == -INFINITY) ? 0.f : m_used;
        // weights 2^(s * scale - m) as bf16 pairs, packed in place (pair j -> sr[j]), then
        // written into the tile's P columns in one TMEM store
        const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(-m_sub, -m_sub);
        float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int i = 0; i < 128; i += 2) {
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), sc2, nm2);
            const float2 p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
            sum2[(i >> 1) & 1] = __fadd2_rn(sum2[(i >> 1) & 1], p);
            sr[i >> 1] = pack_bf16x2(p.x, p.y);
        }
        if (!pv_clear) {
            if (!warp_wait(&S.pv_done[t], (kt - 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
        }
        tmem_st64(t_p, sr);
        tc_wait_st();
        l += (sum2[0].x + sum2[0].y) + (sum2[1].x + sum2[1].y);
        if (zero_v_rows && kt == n_kt - 1 && key0 + kKeyTile > n_keys) {
            // keys at positions >= n_keys hold stale bytes: zero their V rows
            const int s = kt % kVStages;
            if (!warp_wait(&S.v_full[s], (kt / kVStages) & 1)) {
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
            fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.p_full[t]);
    }
    if (ok && warp_wait(&S.pv_done[t], (nt - 1) & 1)) {
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16* orow =
            a.out + (size_t)(row0 + kMmaTokens * t + tl) * kQRowElems + (g * kGroup + hl) * kHeadDim;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(t_o + c * 32, o);
            tc_wait_ld();
            if (row_valid) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(o[8 * j + 0]) * inv, __uint_as_float(o[8 * j + 1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(o[8 * j + 2]) * inv, __uint_as_float(o[8 * j + 3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(o[8 * j + 4]) * inv, __uint_as_float(o[8 * j + 5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(o[8 * j + 6]) * inv, __uint_as_float(o[8 * j + 7]) * inv);
                    *reinterpret_cast<uint4*>(orow + c * 32 + j * 8) = w;
                }
            }
        }
    } else {
        raise_error(a.err, kErrTimeout);
    }
}

__device__ __forceinline__ void prefill_cta(const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                            const CUtensorMap& tmap_v, const PrefillArgs& a, PrefillSmem& S, int tile,
                                            int g) {
    if (tile >= __ldcg(&a.counters[1])) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int4 td = __ldcg(&a.tiles[tile]);
    const int r = td.x, tok0 = td.y, ntok = td.z;
    const int ctx_r = a.ctx[r];
    const int q_len = a.cu[r + 1] - a.cu[r];
    const int row0 = a.cu[r] + tok0;
    const int qpos0 = ctx_r + tok0;
    const int n_keys = ctx_r + q_len;
    const int n_pages = (n_keys + kBlockSize - 1) / kBlockSize;
    const int ntA = min(ntok, kMmaTokens), ntB = max(0, ntok - kMmaTokens);
    const int nA = (qpos0 + ntA - 1) / kKeyTile + 1;
    const int nB = ntB > 0 ? (qpos0 + kMmaTokens + ntB - 1) / kKeyTile + 1 : 0;
    const int n_kt = max(nA, nB);
    const int zero_tile = (nA == n_kt) ? 0 : 1;   // the first MMA tile that reads the last key tile

    if (warp == 1) {
        tmem_alloc(&S.tmem_base, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        mbar_init(&S.q_full, 1);
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&S.k_full[s], 1);
            mbar_init(&S.k_empty[s], 2);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&S.v_full[s], 1);
            mbar_init(&S.v_empty[s], 2);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&S.s_full[s], 1);
            mbar_init(&S.p_full[s], 4);
            mbar_init(&S.pv_done[s], 1);
        }
        mbar_init(&S.s_free[0], 4);
        mbar_init(&S.s_free[1], 4);
        mbar_init(&S.mma_done, 2);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;

    if (warp == 0 || warp == 2) {
        // ---------------------------------------------- TMA producers: K (warp 0), V (warp 2)
        // A key tile is 8 blocks x 2 halves of 64 dims = 16 TMA loads; lane j of the warp
        // issues load j (block j / 2, half j % 2), so a tile's loads leave in one go
        // instead of one after another from a single thread.
        const bool is_k = warp == 0;
        const CUtensorMap* tm = is_k ? &tmap_k : &tmap_v;
        const int nst = is_k ? kKStages : kVStages;
        constexpr int kPages = kKeyTile / kBlockSize;
        const int jb = lane >> 1, jh = lane & 1;          // this lane's block and half (lanes < 16)
        if (lane == 0) prefetch_tmap(tm);
        if (is_k) {
            if (lane == 0) {
                prefetch_tmap(&tmap_q);
                mbar_arrive_expect_tx(&S.q_full, 4 * kHalfBytes);
            }
            __syncwarp();
            if (lane < 4) {
                const int t = lane >> 1, h = lane & 1;
                tma_load_3d(S.q[t][h], &tmap_q, h * 64, g * kGroup, row0 + kMmaTokens * t, &S.q_full);
            }
        }
        const int32_t* trow = a.tables + (size_t)r * a.max_blocks;
        // block-table entry of this lane's block in key tile kt (lanes 0..7 load, the
        // others take it by shuffle), read one tile ahead so its latency overlaps the wait
        // for a free stage
        auto read_entry = [&](int kt) -> int {
            const int pg = kt * kPages + lane;
            const int e = (lane < kPages && kt < n_kt && pg < n_pages) ? trow[pg] : 0;
            return __shfl_sync(0xffffffffu, e, jb & (kPages - 1));
        };
        int next = read_entry(0);
        int issued = 0;
        bool ok = true;
        for (int kt = 0; kt < n_kt; ++kt) {
            const int s = kt % nst;
            const uint32_t ph = (kt / nst) & 1;
            int b = next;
            if ((unsigned)b >= (unsigned)a.num_blocks) {
                if (is_k && jh == 0) raise_error(a.err, kErrBadBlock);
                b = 0;
            }
            const int row = (b * kNumKvHeads + g) * kBlockSize;
            next = read_entry(kt + 1);
            uint64_t* empty = is_k ? &S.k_empty[s] : &S.v_empty[s];
            uint64_t* full = is_k ? &S.k_full[s] : &S.v_full[s];
            ok = __shfl_sync(0xffffffffu, lane == 0 ? (int)mbar_wait(empty, ph ^ 1) : 0, 0) != 0;
            if (!ok) {
                if (lane == 0) raise_error(a.err, kErrTimeout);
                break;
            }
            const int npg = min(kPages, n_pages - kt * kPages);
            if (lane == 0) mbar_arrive_expect_tx(full, npg * kTileBytes);
            __syncwarp();
            if (jb < npg && lane < 2 * kPages) {
                const uint32_t d0 = smem_u32(is_k ? S.k[s][0] : S.v[s][0]);
                tma_load_2d_u32(d0 + jh * kHalfBytes + jb * 2048, tm, jh * 64, row, smem_u32(full));
            }
            ++issued;
        }
        // Drain: wait until every copy issued into this CTA's shared memory landed.
        if (lane == 0) {
            if (is_k && !mbar_wait(&S.q_full, 0)) raise_error(a.err, kErrTimeout);
            for (int kt = issued - nst < 0 ? 0 : issued - nst; kt < issued; ++kt) {
                uint64_t* full = is_k ? &S.k_full[kt % nst] : &S.v_full[kt % nst];
                if (!mbar_wait(full, (kt / nst) & 1)) raise_error(a.err, kErrTimeout);
            }
        }
    } else if (warp == 1 || warp == 3) {
        // ---------------------------------------------------------------- MMA issuers
        // Two groups of MMAs per key tile kt:
        //   X(kt): S = Q_B K_kt^T, then O_A += P_A V_{kt-1}    (issued by warp 1)
        //   Y(kt): S = Q_A K_{kt+1}^T, then O_B += P_B V_{kt-1} (issued by warp 3)
        // Each Q K^T waits until the softmax that read the previous S has loaded it, which
        // it does while the tensor core runs the P V queued behind that Q K^T; a tile's P
        // for key tile kt - 1 is consumed about a round after its S was produced, so the
        // softmax runs off the tensor core's critical path.  A warp that has just queued
        // MMAs sees its next barrier test come back only ~300 cycles later (its shared-
        // memory operations wait behind its tcgen05 ones); with the groups alternating
        // between two warps, the other warp's group keeps the tensor core busy meanwhile.
        // Each warp runs its loop in step (waits, descriptor arithmetic: values the same
        // in every lane), and one elected lane issues each tcgen05 instruction.
        const bool xw = warp == 1;
        const bool leader = elect_one();
        constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, 0);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, 1);
        // Descriptors are built once: Q tiles, K stages and V stages are 32 KiB apart
        // and a K step moves 32 bytes inside the swizzle rows (or to the next 64-dim
        // half), so every MMA's operands are a constant step from these bases (the
        // 14-bit address field never carries: shared addresses stay below 227 KiB).
        constexpr uint64_t kStep32K = (2 * kHalfBytes) >> 4;
        const uint64_t q_desc0 = smem_desc_sw128(smem_u32(S.q[0][0]), 16, 1024);
        const uint64_t k_desc0 = smem_desc_sw128(smem_u32(S.k[0][0]), 16, 1024);
        const uint64_t v_desc0 = smem_desc_sw128(smem_u32(S.v[0][0]), kHalfBytes, 1024);
        bool ok = warp_wait(&S.q_full, 0);
        // The S buffer's uses in order: Q_A K_0^T, Q_B K_0^T, Q_A K_1^T, ... (only tile A's
        // when tile B is empty; tile B may have one key tile more than A).  Each Q K^T waits
        // until the softmax that read the previous use has loaded it: phase j of s_free[t]
        // is tile t's j-th read.  A warp only ever waits for the phase after one it has
        // already seen complete, so a parity test cannot be satisfied by an older phase.
        //   Q_B K_kt^T: s_free[0] phase kt (kt < nA), else s_free[1] phase kt - 1;
        //   Q_A K_kt^T (kt >= 1): s_free[1] phase kt - 1 (tile B not empty), else s_free[0].
        auto s_bar_b = [&](int kt) { return kt < nA ? &S.s_free[0] : &S.s_free[1]; };
        auto s_ph_b = [&](int kt) { return (uint32_t)((kt < nA ? kt : kt - 1) & 1); };
        auto s_bar_a = [&]() { return nB > 0 ? &S.s_free[1] : &S.s_free[0]; };
        auto wait_k = [&](int kt) -> bool { return warp_wait(&S.k_full[kt % kKStages], (kt / kKStages) & 1); };
        auto wait_p = [&](int t, int kt) -> bool { return warp_wait(&S.p_full[t], kt & 1); };
        auto wait_v = [&](int kt) -> bool { return warp_wait(&S.v_full[kt % kVStages], (kt / kVStages) & 1); };
        auto test_k = [&](int kt) { return mbar_test(&S.k_full[kt % kKStages], (kt / kKStages) & 1); };
        auto test_p = [&](int t, int kt) { return mbar_test(&S.p_full[t], kt & 1); };
        auto test_v = [&](int kt) { return mbar_test(&S.v_full[kt % kVStages], (kt / kVStages) & 1); };
        // K and V stages are released by two commits (k_empty / v_empty count 2): one per
        // tile that reads the stage, or two by the only one (each commit tracks only the
        // committing thread's MMAs).
        auto mma_qk = [&](int t, int kt) {
            const int s = kt % kKStages;
            const uint64_t qa = q_desc0 + (uint64_t)t * kStep32K, kb = k_desc0 + (uint64_t)s * kStep32K;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t koff = (uint64_t)((((kk >> 2) * kHalfBytes) + (kk & 3) * 32) >> 4);
                    tc_mma_f16(tmem, qa + koff, kb + koff, idesc_qk, kk > 0 ? 1u : 0u);
                }
                tc_commit(&S.s_full[t]);
                tc_commit(&S.k_empty[s]);
                if (kt >= (t ? nA : nB)) tc_commit(&S.k_empty[s]);
            }
            __syncwarp();
        };
        auto mma_pv = [&](int t, int kt) {
            const int s = kt % kVStages;
            const uint64_t vb = v_desc0 + (uint64_t)s * kStep32K;
            const uint32_t d = tmem + 256 + t * 128, pa = tmem + 128 + t * 64;
            const uint32_t acc0 = kt > 0 ? 1u : 0u;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc_mma_f16_ts(d, pa + kk * 8, vb + (uint64_t)((kk * 2048) >> 4), idesc_pv, kk > 0 ? 1u : acc0);
                tc_commit(&S.pv_done[t]);
                tc_commit(&S.v_empty[s]);
                if (kt >= (t ? nA : nB)) tc_commit(&S.v_empty[s]);
            }
            __syncwarp();
        };
        // The last key tile's V rows past the keys are zeroed by one tile's softmax before
        // it announces P; the other tile's P V of that key tile waits for that P too.
        const int last = n_kt - 1;
        auto zero_wait = [&](int t, int kt) { return kt == last && t != zero_tile; };
        // A group's barriers are tested together first (one round trip instead of one per
        // barrier); only if one of them is not complete yet does the warp wait on them in
        // turn, the S barrier (normally the last to complete) last, so that the MMAs go
        // out right after the softmax has read S.
        if (xw) {
            for (int kt = 0; kt <= n_kt && ok; ++kt) {
                const bool qk = kt < nB, pv = kt >= 1 && kt <= nA;
                if (!qk && !pv) continue;
                const bool zw = pv && zero_wait(0, kt - 1);
                const uint32_t ready = (qk ? (kt < nA ? 1u : test_k(kt)) & mbar_test(s_bar_b(kt), s_ph_b(kt)) : 1u) &
                                       (pv ? test_p(0, kt - 1) & test_v(kt - 1) : 1u) & (zw ? test_p(1, kt - 1) : 1u);
                if (!__all_sync(0xffffffffu, ready != 0) &&
                    !(ok = (!pv || (wait_p(0, kt - 1) && wait_v(kt - 1))) && (!zw || wait_p(1, kt - 1)) &&
                           (!qk || ((kt < nA || wait_k(kt)) && warp_wait(s_bar_b(kt), s_ph_b(kt))))))
                    break;
                tc_fence_after();
                if (qk) mma_qk(1, kt);
                if (pv) mma_pv(0, kt - 1);
            }
        } else {
            if (ok && nA > 0 && (ok = wait_k(0))) {
                tc_fence_after();
                mma_qk(0, 0);
            }
            for (int kt = 0; kt <= n_kt && ok; ++kt) {
                const bool qk = kt + 1 < nA, pv = kt >= 1 && kt <= nB;
                if (!qk && !pv) continue;
                const bool zw = pv && zero_wait(1, kt - 1);
                const uint32_t ready = (qk ? test_k(kt + 1) & mbar_test(s_bar_a(), kt & 1) : 1u) &
                                       (pv ? test_p(1, kt - 1) & test_v(kt - 1) : 1u) & (zw ? test_p(0, kt - 1) : 1u);
                if (!__all_sync(0xffffffffu, ready != 0) &&
                    !(ok = (!pv || (wait_p(1, kt - 1) && wait_v(kt - 1))) && (!zw || wait_p(0, kt - 1)) &&
                           (!qk || (wait_k(kt + 1) && warp_wait(s_bar_a(), kt & 1)))))
                    break;
                tc_fence_after();
                if (qk) mma_qk(0, kt + 1);
                if (pv) mma_pv(1, kt - 1);
            }
        }
        if (!ok && leader) raise_error(a.err, kErrTimeout);
        // No MMA may still be running when TMEM is released (mma_done: one commit per warp).
        if (leader) tc_commit(&S.mma_done);
        __syncwarp();
        if (!warp_wait(&S.mma_done, 0) && leader) raise_error(a.err, kErrTimeout);
    } else if (warp >= 4) {
        // --------------------------------------------------------- softmax + epilogue
        const int t = (warp - 4) >> 2;
        const int nt = t ? nB : nA;
        if (nt > 0)
            softmax_tile(S, a, tmem, t, warp & 3, lane, g, row0, qpos0, t ? ntB : ntA, nt, n_kt, n_keys,
                         t == zero_tile);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// The prefill kernel's arguments for one step.
inline PrefillArgs make_prefill_args(const StepArgs& a) {
    const StepLayout& L = a.lay;
    PrefillArgs pa;
    pa.counters = reinterpret_cast<const int32_t*>(a.ws + L.counters_off);
    pa.done = reinterpret_cast<int32_t*>(a.ws + L.counters_off) + 3;
    pa.tiles = reinterpret_cast<const int4*>(a.ws + L.prefill_tiles_off);
    pa.cu = a.cu_seqlens_q;
    pa.ctx = a.context_lens;
    pa.tables = a.block_tables;
    pa.max_blocks = a.max_blocks_per_seq;
    pa.num_blocks = a.num_blocks;
    pa.out = static_cast<__nv_bfloat16*>(a.out);
    pa.err = a.err;
    pa.scale_log2 = a.softmax_scale * 1.4426950408889634f;
    return pa;
}

}  // namespace
}  // namespace kvp
