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
// Work item = one (request, 64-token q tile, KV head g), split into two MMA tiles A and B
// of 32 tokens each.  The 128 rows of an MMA tile are its 32 tokens x the 4 query heads
// that share KV head g (row = 4 * token + head), so every K/V tile is loaded once for the
// whole GQA group and serves both MMA tiles.  Key tiles are 128 keys = 8 blocks of 16:
// each block's (block, head g) 4 KiB tile is fetched by two 2-D TMA loads (one per 64-dim
// half, 128-byte swizzle), landing in the canonical K-major SW128 layout.
//
// A CTA takes items one after another from a device counter, in the metadata kernel's
// longest-first order, until none are left (in the mixed step kernel, after the decode
// range its ticket may give it).  The rings, barriers and TMEM carry over from item to item
// and every role runs ahead into the next item as soon as its part of the current one is
// done, so a CTA pays its start-up (TMEM, barriers, the first loads) once.
//
// Warp roles (12 warps): warp 0 claims items (into a 2-deep ring that the other roles
// read) and issues the TMA loads of Q and of K tiles into a 3-stage ring, warp 2 those of
// V tiles into a 2-stage ring; warps 1 and 3 issue the MMAs (warp 1 owns TMEM); warps 4-7
// run the softmax of tile A and warps 8-11 that of tile B, one thread per MMA row (TMEM
// lane).  TMEM (512 columns): one S buffer shared by the two tiles at 0, P of A at 128 and
// of B at 192 (bf16 pairs, 64 columns each), O of A at 256 and of B at 384.  With P in
// columns of its own, S is free again as soon as a softmax has loaded it into registers,
// so the next Q K^T need not wait for the P V of the same tile.  Per key tile a softmax
// thread: reads its whole S row from TMEM in one load and frees S,
// keeps a running max m in base 2 (scores x softmax_scale x log2 e) that moves only when
// the tile's max exceeds it by more than 8 (then O and l are rescaled in place, after the
// tile's previous P V has completed: until then weights stay below 2^8, which bf16 and
// fp32 hold exactly enough), writes P = 2^(s - m) as bf16 pairs into its P columns (once
// the previous P V has read them), and the P V MMA reads P from TMEM as its A operand (V
// from shared memory, MN-major: keys are the K dimension).
// End of an item: O / l rounded to bf16 for the tile's valid rows; the tile's next P V
// (the next item's first, which overwrites O) waits for the next P, which the same
// threads publish only after reading O.
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

static_assert(kPrefillTileTokens == 2 * kMmaTokens, "a work item is two MMA tiles");

constexpr int kItemSlots = 2;
constexpr int kItemReaders = 11;   // warps that read an item: V, the two MMA warps, 8 softmax warps

// One work item as warp 0 describes it to the other roles.
struct PrefillItem {
    int r;           // request (-1: no more items)
    int g;           // KV head
    int row0;        // packed row of the item's first token
    int qpos0;       // that token's position in its request
    int n_keys;      // keys the item's last token sees (context + chunk rows)
    int n_pages;     // blocks that hold them
    int ntA, ntB;    // tokens of MMA tiles A and B
    int nA, nB;      // key tiles that tiles A and B read (nB is 0, nA or nA + 1)
    int n_kt;        // key tiles of the item
    int zero_tile;   // the tile whose softmax zeroes the last key tile's stale V rows
};

struct __align__(1024) PrefillSmem {
    uint8_t q[2][2][kHalfBytes];     // [MMA tile][d half][128 rows]
    uint8_t k[kKStages][2][kHalfBytes];   // [stage][d half][128 keys]
    uint8_t v[kVStages][2][kHalfBytes];   // [stage][d half][128 keys]
    PrefillItem item[kItemSlots];
    uint64_t item_full[kItemSlots], item_empty[kItemSlots];
    uint64_t q_full[2], q_empty[2];       // per MMA tile
    uint64_t k_full[kKStages], k_empty[kKStages];
    uint64_t v_full[kVStages], v_empty[kVStages];
    uint64_t s_full[2], p_full[2], pv_done[2];   // per MMA tile
    // A softmax has read S: [0] before the next Q_B K^T (warp 1 waits), [1] before the
    // next Q_A K^T (warp 3 waits).
    uint64_t s_free[2];
    uint64_t mma_done;
    uint32_t tmem_base;
};

struct PrefillArgs {
    const int32_t* counters;
    int32_t* done;               // CTAs that have finished (zeroed by the metadata kernel)
    int32_t* next_item;          // items claimed (zeroed by the metadata kernel)
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

// Item k (tile k / 8 of the metadata kernel's list, KV head k % 8); r = -1 past the end.
__device__ __forceinline__ PrefillItem describe_item(const PrefillArgs& a, int k, int n_items) {
    PrefillItem it{};
    it.r = -1;
    if (k < 0 || k >= n_items) return it;
    const int4 td = __ldcg(&a.tiles[k / kNumKvHeads]);
    const int r = td.x, tok0 = td.y, ntok = td.z;
    const int ctx_r = a.ctx[r];
    const int cu0 = a.cu[r], q_len = a.cu[r + 1] - cu0;
    it.r = r;
    it.g = k % kNumKvHeads;
    it.row0 = cu0 + tok0;
    it.qpos0 = ctx_r + tok0;
    it.n_keys = ctx_r + q_len;
    it.n_pages = (it.n_keys + kBlockSize - 1) / kBlockSize;
    it.ntA = min(ntok, kMmaTokens);
    it.ntB = max(0, ntok - kMmaTokens);
    it.nA = (it.qpos0 + it.ntA - 1) / kKeyTile + 1;
    it.nB = it.ntB > 0 ? (it.qpos0 + kMmaTokens + it.ntB - 1) / kKeyTile + 1 : 0;
    it.n_kt = max(it.nA, it.nB);
    it.zero_tile = (it.nA == it.n_kt) ? 0 : 1;
    return it;
}

// Item i of this CTA from its ring slot (whole warp); then frees the slot's copy.
__device__ __forceinline__ bool read_item(PrefillSmem& S, int i, int lane, PrefillItem& it) {
    const int slot = i % kItemSlots;
    if (!warp_wait(&S.item_full[slot], (uint32_t)((i / kItemSlots) & 1))) return false;
    it = S.item[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.item_empty[slot]);
    return true;
}

// Softmax and epilogue of one MMA tile of one item (a warpgroup, one thread per row).
// sf = this tile's Q K^T (and P V) of earlier items: the phase base of s_full[t],
// p_full[t] and pv_done[t]; kb = key tiles of earlier items (the V ring position).
__device__ __forceinline__ bool softmax_tile(PrefillSmem& S, const PrefillArgs& a, uint32_t tmem, int t, int wq,
                                             int lane, const PrefillItem& it, int sf, int kb) {
    const int nt = t ? it.nB : it.nA;
    const int row = wq * 32 + lane;
    const int tl = row >> 2, hl = row & 3;
    const bool row_valid = tl < (t ? it.ntB : it.ntA);
    const int tq0 = it.qpos0 + kMmaTokens * t;       // position of the tile's first token
    const int qpos = row_valid ? tq0 + tl : -1;
    const bool zero_v_rows = t == it.zero_tile;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off;
    const uint32_t t_p = tmem + 128 + t * 64 + lane_off;
    const uint32_t t_o = tmem + 256 + t * 128 + lane_off;
    const float sc = a.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int kt = 0; kt < nt; ++kt) {
        if (!warp_wait(&S.s_full[t], (sf + kt) & 1)) {
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
        // the next use of S: after Q_A K_kt^T comes Q_B K_kt^T if tile B reads key tile kt,
        // else a Q_A K^T; after Q_B K_kt^T comes Q_A K_{kt+1}^T, or tile B's extra key
        // tile, or the next item's first Q_A K^T
        const int next_b = t == 0 ? (kt < it.nB) : (kt + 1 >= it.nA && kt + 1 < it.nB);
        if (lane == 0) mbar_arrive(&S.s_free[next_b ? 0 : 1]);
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
                if (!warp_wait(&S.pv_done[t], (sf + kt - 1) & 1)) {
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
            if (!warp_wait(&S.pv_done[t], (sf + kt - 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
        }
        tmem_st64(t_p, sr);
        tc_wait_st();
        l += (sum2[0].x + sum2[0].y) + (sum2[1].x + sum2[1].y);
        if (zero_v_rows && kt == it.n_kt - 1 && key0 + kKeyTile > it.n_keys) {
            // keys at positions >= n_keys hold stale bytes: zero their V rows
            const int s = (kb + kt) % kVStages;
            if (!warp_wait(&S.v_full[s], ((kb + kt) / kVStages) & 1)) {
                ok = false;
                break;
            }
            if (key0 + row >= it.n_keys) {
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
    if (ok && warp_wait(&S.pv_done[t], (sf + nt - 1) & 1)) {
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16* orow =
            a.out + (size_t)(it.row0 + kMmaTokens * t + tl) * kQRowElems + (it.g * kGroup + hl) * kHeadDim;
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
        return true;
    }
    raise_error(a.err, kErrTimeout);
    return false;
}

// The CTA body: items from first_item (if >= 0), then from the counter next_item (if
// not null) until it runs past the step's items.
__device__ __forceinline__ void prefill_cta(const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                            const CUtensorMap& tmap_v, const PrefillArgs& a, PrefillSmem& S,
                                            int first_item, int32_t* next_item) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 1) {
        tmem_alloc(&S.tmem_base, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kItemSlots; ++s) {
            mbar_init(&S.item_full[s], 1);
            mbar_init(&S.item_empty[s], kItemReaders);
        }
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&S.k_full[s], 1);
            mbar_init(&S.k_empty[s], 2);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&S.v_full[s], 1);
            mbar_init(&S.v_empty[s], 2);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&S.q_full[s], 1);
            mbar_init(&S.q_empty[s], 1);
            mbar_init(&S.s_full[s], 1);
            mbar_init(&S.p_full[s], 4);
            mbar_init(&S.pv_done[s], 1);
            mbar_init(&S.s_free[s], 4);
        }
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
        // instead of one after another from a single thread.  Warp 0 also claims the
        // items and loads each item's Q tiles, each once the previous item's last Q K^T
        // of that tile has read it.
        const bool is_k = warp == 0;
        const CUtensorMap* tm = is_k ? &tmap_k : &tmap_v;
        const int nst = is_k ? kKStages : kVStages;
        constexpr int kPages = kKeyTile / kBlockSize;
        const int jb = lane >> 1, jh = lane & 1;          // this lane's block and half (lanes < 16)
        if (lane == 0) {
            prefetch_tmap(tm);
            if (is_k) prefetch_tmap(&tmap_q);
        }
        const int n_items = is_k ? __ldcg(&a.counters[1]) * kNumKvHeads : 0;
        int kg = 0;      // key tiles issued into the ring so far
        int items = 0;   // items whose loads were issued
        bool ok = true;
        for (int i = 0; ok; ++i) {
            PrefillItem it;
            if (is_k) {
                int k = -1;
                if (lane == 0)
                    k = (i == 0 && first_item >= 0) ? first_item : (next_item != nullptr ? atomicAdd(next_item, 1) : -1);
                it = describe_item(a, __shfl_sync(0xffffffffu, k, 0), n_items);
                const int slot = i % kItemSlots;
                if (i >= kItemSlots &&
                    !(ok = warp_wait(&S.item_empty[slot], (uint32_t)(((i / kItemSlots) - 1) & 1))))
                    break;
                if (lane == 0) {
                    S.item[slot] = it;
                    mbar_arrive(&S.item_full[slot]);   // releases the description to its readers
                }
                __syncwarp();
            } else if (!(ok = read_item(S, i, lane, it))) {
                break;
            }
            if (it.r < 0) break;
            ++items;
            auto load_q = [&](int t) -> bool {
                if (i > 0 && !warp_wait(&S.q_empty[t], (uint32_t)((i - 1) & 1))) return false;
                if (lane == 0) mbar_arrive_expect_tx(&S.q_full[t], 2 * kHalfBytes);
                __syncwarp();
                if (lane < 2)
                    tma_load_3d(S.q[t][lane], &tmap_q, lane * 64, it.g * kGroup, it.row0 + kMmaTokens * t, &S.q_full[t]);
                return true;
            };
            const int32_t* trow = a.tables + (size_t)it.r * a.max_blocks;
            // block-table entry of this lane's block in key tile kt (lanes 0..7 load, the
            // others take it by shuffle), read one tile ahead so its latency overlaps the
            // wait for a free stage
            auto read_entry = [&](int kt) -> int {
                const int pg = kt * kPages + lane;
                const int e = (lane < kPages && kt < it.n_kt && pg < it.n_pages) ? trow[pg] : 0;
                return __shfl_sync(0xffffffffu, e, jb & (kPages - 1));
            };
            int next = read_entry(0);
            for (int kt = 0; kt < it.n_kt; ++kt, ++kg) {
                if (is_k && kt == 0 && !(ok = load_q(0))) break;
                const int s = kg % nst;
                const uint32_t ph = (kg / nst) & 1;
                int b = next;
                if ((unsigned)b >= (unsigned)a.num_blocks) {
                    if (is_k && jh == 0) raise_error(a.err, kErrBadBlock);
                    b = 0;
                }
                const int row = (b * kNumKvHeads + it.g) * kBlockSize;
                next = read_entry(kt + 1);
                uint64_t* empty = is_k ? &S.k_empty[s] : &S.v_empty[s];
                uint64_t* full = is_k ? &S.k_full[s] : &S.v_full[s];
                if (kg >= nst && !(ok = warp_wait(empty, ph ^ 1))) break;
                const int npg = min(kPages, it.n_pages - kt * kPages);
                if (lane == 0) mbar_arrive_expect_tx(full, npg * kTileBytes);
                __syncwarp();
                if (jb < npg && lane < 2 * kPages) {
                    const uint32_t d0 = smem_u32(is_k ? S.k[s][0] : S.v[s][0]);
                    tma_load_2d_u32(d0 + jh * kHalfBytes + jb * 2048, tm, jh * 64, row, smem_u32(full));
                }
                if (is_k && kt == 0 && !(ok = load_q(1))) {
                    ++kg;
                    break;
                }
            }
        }
        if (!ok && lane == 0) raise_error(a.err, kErrTimeout);
        // Drain: wait until every copy issued into this CTA's shared memory landed.
        if (lane == 0) {
            if (is_k && items > 0)
                for (int t = 0; t < 2; ++t)
                    if (!mbar_wait(&S.q_full[t], (uint32_t)((items - 1) & 1))) raise_error(a.err, kErrTimeout);
            for (int j = kg - nst < 0 ? 0 : kg - nst; j < kg; ++j) {
                uint64_t* full = is_k ? &S.k_full[j % nst] : &S.v_full[j % nst];
                if (!mbar_wait(full, (j / nst) & 1)) raise_error(a.err, kErrTimeout);
            }
        }
    } else if (warp == 1 || warp == 3) {
        // ---------------------------------------------------------------- MMA issuers
        // Two groups of MMAs per key tile kt of an item:
        //   X(kt): S = Q_B K_kt^T, then O_A += P_A V_{kt-1}    (issued by warp 1)
        //   Y(kt): S = Q_A K_{kt+1}^T, then O_B += P_B V_{kt-1} (issued by warp 3)
        // after S = Q_A K_0^T (warp 3).  Each Q K^T waits until the softmax that read the
        // previous S has loaded it, which it does while the tensor core runs the P V queued
        // behind that Q K^T; a tile's P for key tile kt - 1 is consumed about a round after
        // its S was produced, so the softmax runs off the tensor core's critical path.  A
        // warp that has just queued MMAs sees its next barrier test come back only ~300
        // cycles later (its shared-memory operations wait behind its tcgen05 ones); with the
        // groups alternating between two warps, the other warp's group keeps the tensor core
        // busy meanwhile.  Each warp runs its loop in step (waits, descriptor arithmetic:
        // values the same in every lane), and one elected lane issues each tcgen05
        // instruction.
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
        // Counts over this CTA's earlier items: key tiles (the K and V ring positions), P
        // of tiles A and B (the p_full phases), and the Q K^T this warp issued (the phases
        // of its s_free barrier: each Q_B K^T waits s_free[0] phase = Q_B K^T before it,
        // each Q_A K^T but the CTA's first s_free[1] phase = Q_A K^T before it - 1).  Every
        // barrier a warp waits on, it waits on phase after phase, so a parity test cannot
        // be satisfied by an older phase.
        int kb = 0, pa = 0, pb = 0, nq = 0;
        PrefillItem it{};
        auto k_bar = [&](int kt) { return &S.k_full[(kb + kt) % kKStages]; };
        auto k_ph = [&](int kt) { return (uint32_t)(((kb + kt) / kKStages) & 1); };
        auto v_bar = [&](int kt) { return &S.v_full[(kb + kt) % kVStages]; };
        auto v_ph = [&](int kt) { return (uint32_t)(((kb + kt) / kVStages) & 1); };
        auto p_ph = [&](int t, int kt) { return (uint32_t)(((t ? pb : pa) + kt) & 1); };
        // K and V stages are released by two commits (k_empty / v_empty count 2): one per
        // tile that reads the stage, or two by the only one (each commit tracks only the
        // committing thread's MMAs).
        auto mma_qk = [&](int t, int kt) {
            const int s = (kb + kt) % kKStages;
            const uint64_t qa = q_desc0 + (uint64_t)t * kStep32K, kd = k_desc0 + (uint64_t)s * kStep32K;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t koff = (uint64_t)((((kk >> 2) * kHalfBytes) + (kk & 3) * 32) >> 4);
                    tc_mma_f16(tmem, qa + koff, kd + koff, idesc_qk, kk > 0 ? 1u : 0u);
                }
                tc_commit(&S.s_full[t]);
                tc_commit(&S.k_empty[s]);
                if (kt >= (t ? it.nA : it.nB)) tc_commit(&S.k_empty[s]);
                if (kt == (t ? it.nB : it.nA) - 1) tc_commit(&S.q_empty[t]);   // the item's last read of Q_t
            }
            __syncwarp();
            ++nq;
        };
        auto mma_pv = [&](int t, int kt) {
            const int s = (kb + kt) % kVStages;
            const uint64_t vd = v_desc0 + (uint64_t)s * kStep32K;
            const uint32_t d = tmem + 256 + t * 128, pt = tmem + 128 + t * 64;
            const uint32_t acc0 = kt > 0 ? 1u : 0u;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc_mma_f16_ts(d, pt + kk * 8, vd + (uint64_t)((kk * 2048) >> 4), idesc_pv, kk > 0 ? 1u : acc0);
                tc_commit(&S.pv_done[t]);
                tc_commit(&S.v_empty[s]);
                if (kt >= (t ? it.nA : it.nB)) tc_commit(&S.v_empty[s]);
            }
            __syncwarp();
        };
        bool ok = true;
        // A group's barriers are tested together first (one round trip instead of one per
        // barrier); only if one of them is not complete yet does the warp wait on them in
        // turn, the S barrier (normally the last to complete) last, so that the MMAs go
        // out right after the softmax has read S.
        for (int i = 0; ok; ++i) {
            if (!(ok = read_item(S, i, lane, it)) || it.r < 0) break;
            const int nA = it.nA, nB = it.nB, n_kt = it.n_kt, last = n_kt - 1;
            const uint32_t qph = (uint32_t)(i & 1);
            if (xw) {
                for (int kt = 0; kt <= n_kt && ok; ++kt) {
                    const bool qk = kt < nB, pv = kt >= 1 && kt <= nA, q0 = kt == 0;
                    // the other tile's P of the last key tile, whose softmax zeroed V's stale rows
                    const bool zw = pv && kt - 1 == last && it.zero_tile == 1;
                    if (!qk && !pv && !q0) continue;
                    const uint32_t ready =
                        (q0 ? mbar_test(&S.q_full[1], qph) : 1u) &
                        (qk ? (kt < nA ? 1u : mbar_test(k_bar(kt), k_ph(kt))) & mbar_test(&S.s_free[0], nq & 1) : 1u) &
                        (pv ? mbar_test(&S.p_full[0], p_ph(0, kt - 1)) & mbar_test(v_bar(kt - 1), v_ph(kt - 1)) : 1u) &
                        (zw ? mbar_test(&S.p_full[1], p_ph(1, kt - 1)) : 1u);
                    if (!__all_sync(0xffffffffu, ready != 0) &&
                        !(ok = (!pv || (warp_wait(&S.p_full[0], p_ph(0, kt - 1)) &&
                                        warp_wait(v_bar(kt - 1), v_ph(kt - 1)))) &&
                               (!zw || warp_wait(&S.p_full[1], p_ph(1, kt - 1))) &&
                               (!q0 || warp_wait(&S.q_full[1], qph)) &&
                               (!qk || ((kt < nA || warp_wait(k_bar(kt), k_ph(kt))) &&
                                        warp_wait(&S.s_free[0], nq & 1)))))
                        break;
                    tc_fence_after();
                    if (qk) mma_qk(1, kt);
                    if (pv) mma_pv(0, kt - 1);
                    if (q0 && nB == 0) {   // tile B is empty: its Q tile is free at once
                        if (leader) tc_commit(&S.q_empty[1]);
                        __syncwarp();
                    }
                }
            } else {
                // S = Q_A K_0^T (after the previous item's last use of S)
                {
                    const uint32_t ready = mbar_test(&S.q_full[0], qph) & mbar_test(k_bar(0), k_ph(0)) &
                                           (nq > 0 ? mbar_test(&S.s_free[1], (nq - 1) & 1) : 1u);
                    if (!__all_sync(0xffffffffu, ready != 0) &&
                        !(ok = warp_wait(&S.q_full[0], qph) && warp_wait(k_bar(0), k_ph(0)) &&
                               (nq == 0 || warp_wait(&S.s_free[1], (nq - 1) & 1))))
                        break;
                    tc_fence_after();
                    mma_qk(0, 0);
                }
                for (int kt = 0; kt <= n_kt && ok; ++kt) {
                    const bool qk = kt + 1 < nA, pv = kt >= 1 && kt <= nB;
                    const bool zw = pv && kt - 1 == last && it.zero_tile == 0;
                    if (!qk && !pv) continue;
                    const uint32_t ready =
                        (qk ? mbar_test(k_bar(kt + 1), k_ph(kt + 1)) & mbar_test(&S.s_free[1], (nq - 1) & 1) : 1u) &
                        (pv ? mbar_test(&S.p_full[1], p_ph(1, kt - 1)) & mbar_test(v_bar(kt - 1), v_ph(kt - 1)) : 1u) &
                        (zw ? mbar_test(&S.p_full[0], p_ph(0, kt - 1)) : 1u);
                    if (!__all_sync(0xffffffffu, ready != 0) &&
                        !(ok = (!pv || (warp_wait(&S.p_full[1], p_ph(1, kt - 1)) &&
                                        warp_wait(v_bar(kt - 1), v_ph(kt - 1)))) &&
                               (!zw || warp_wait(&S.p_full[0], p_ph(0, kt - 1))) &&
                               (!qk || (warp_wait(k_bar(kt + 1), k_ph(kt + 1)) &&
                                        warp_wait(&S.s_free[1], (nq - 1) & 1)))))
                        break;
                    tc_fence_after();
                    if (qk) mma_qk(0, kt + 1);
                    if (pv) mma_pv(1, kt - 1);
                }
            }
            kb += n_kt;
            pa += nA;
            pb += nB;
        }
        if (!ok && leader) raise_error(a.err, kErrTimeout);
        // No MMA may still be running when TMEM is released (mma_done: one commit per warp).
        if (leader) tc_commit(&S.mma_done);
        __syncwarp();
        if (!warp_wait(&S.mma_done, 0) && leader) raise_error(a.err, kErrTimeout);
    } else if (warp >= 4) {
        // --------------------------------------------------------- softmax + epilogue
        const int t = (warp - 4) >> 2;
        int sf = 0, kb = 0;   // this tile's Q K^T and the key tiles of earlier items
        PrefillItem it;
        for (int i = 0;; ++i) {
            if (!read_item(S, i, lane, it)) {
                raise_error(a.err, kErrTimeout);
                break;
            }
            if (it.r < 0) break;
            const int nt = t ? it.nB : it.nA;
            if (nt > 0 && !softmax_tile(S, a, tmem, t, warp & 3, lane, it, sf, kb)) break;
            sf += nt;
            kb += it.n_kt;
        }
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
    pa.next_item = reinterpret_cast<int32_t*>(a.ws + L.counters_off) + 6;
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
