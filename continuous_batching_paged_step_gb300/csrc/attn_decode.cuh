// Device code of the decode rows' split-KV attention, shared by the decode kernel and the
// mixed step kernel (included by attn_decode.cu and attn_mixed.cu).
//
// Decode rows (q_len == 1): split-KV paged attention, HBM-bound.
//
// The decode formula of page "Continuous Batching" (k4i.top), section "与 KV cache 的关
// 系": the row's query attends to [K_cache; k_t] and [V_cache; v_t] of its own request,
// i.e. all positions 0 .. ctx of that request (this step's key was appended already).
// Decode streams the whole KV history every step (same page, section "为什么 decode 是
// bandwidth-bound"), so the kernel is built to keep HBM busy:
//
// * Work: the 16-token blocks of all decode rows, concatenated in request order
//   (page_off[r] = first global block of request r), are cut into equal contiguous
//   ranges, one per CTA (one CTA per SM of the decode's share of the SMs, which the step's
//   metadata kernel sizes so that the prefill tiles run on the others; fewer CTAs when
//   there are under 4 blocks per CTA; more, in whole waves, when a range would exceed the
//   1,024 blocks a CTA stages).  SMs do not all get the same share of HBM bandwidth (on
//   a GB300 some SMs finish equal ranges up to ~20 % later, the same SMs every step), so
//   each range keeps only its first 80 % as the CTA's own part; its last 20 % is cut into
//   a few chunks that any CTA takes, through one global counter, once its own part is
//   issued.  Fast SMs so take more chunks and all CTAs end together.
// * Pieces (own parts and chunks) are numbered densely in sequence order.  A request cut
//   by piece boundaries produces one partial per piece (slot r + piece), which the
//   combine kernel after the step's attention kernels merges; a request inside one piece
//   is finished in place.
// * One producer warp per CTA issues all copies: the block ids, requests and positions
//   of the own part are looked up by the whole CTA up front (into shared memory), those
//   of a chunk by a scheduler warp, which claims the chunk when the producer asks (a few
//   blocks before it runs out of work) while earlier blocks stream.  One block of all 8
//   KV heads is 128 rows (head x token) of 128 dims in the pool, so its K and its V
//   arrive with four tensor-map loads (one per 64-dim half, 128-byte swizzle) into a
//   3-stage ring of 64 KiB stages; with each stage the producer hands the consumers the
//   block's request, position and segment flags.
// * One consumer warp per KV head.  Its 4 query heads share every K/V byte (GQA
//   packing), and the two contractions of a block are small matrix products, which run
//   on the tensor cores (mma.sync m16n8k16, bf16 operands, fp32 accumulation) instead
//   of as thousands of scalar FMAs:  S^T = K Q^T (16 tokens x 8 columns, the 4 query
//   heads and 4 zero columns) and O^T += V^T P^T (128 dims x 8 columns).  K and V
//   fragments come from the swizzled tiles with ldmatrix (V transposed on the way), so
//   reads are free of bank conflicts; the weights go from the score fragment to the
//   P^T operand with one register transpose (movmatrix) per 8 tokens.  A warp reads all
//   of its fragments of a block first and releases the stage at once.
// * Online softmax in base 2 (scores x softmax_scale x log2 e) against a reference max
//   per head that moves only when a score exceeds it by more than 2^8 (a warp vote; the
//   max reduction and the rescale run only then), with per-lane partial sums reduced
//   once per segment.  Weights enter P.V rounded to bf16; the sums use them unrounded.
// Partial results keep (m, l, unnormalised acc); the merge computes
// O = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s with M = max_s m_s.
// Keys at positions >= ctx + 1 of the last block are excluded: score -inf, and their V
// values zeroed in the fragments (stale bytes could hold NaN, and 0 x NaN is NaN).
#pragma once

#include <cuda.h>

#include "kvp_device.cuh"
#include "kvp_launch.h"

namespace kvp {

namespace {

constexpr int kConsumerWarps = kNumKvHeads;   // one per KV head
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kSchedulerWarp = kConsumerWarps + 1;
constexpr int kDecThreads = (kConsumerWarps + 2) * 32;   // + the producer and the scheduler warp
constexpr int kDecStages = 3;
constexpr int kBlockRows = kNumKvHeads * kBlockSize;   // rows (head, token) of one block: 128
constexpr int kHalfTile = kBlockRows * 128;            // one block's 64-dim half: 128 rows x 128 B
constexpr int kStageBytes = 4 * kHalfTile;             // K and V, two halves each: 64 KiB

constexpr int kIdCap = 1024;       // blocks of a CTA's range (its own part is staged up front)
constexpr int kTailPercent = 20;   // share of each range handed out as chunks
constexpr int kChunkTarget = 8;    // blocks per chunk, at least (fewer pieces to merge; 4 and 6 measured slower)
constexpr int kMaxPieces = 8;      // pieces per range: own part + chunks
constexpr int kMaxChunk = 32;      // blocks per chunk, at most (one scheduler lane each)
constexpr int kClaimLead = 3;      // blocks still to issue (own part or chunk) when the next chunk is claimed
constexpr int kPageOffCap = 2047;  // requests whose block offsets a CTA stages in shared memory

// segment flags next to a block's position in its request
constexpr uint32_t kPosMask = 0x00FFFFFFu;
constexpr uint32_t kFirst = 1u << 24;   // first block of a segment (request x piece)
constexpr uint32_t kLast = 1u << 25;    // last block of a segment
constexpr uint32_t kWhole = 1u << 26;   // the segment is the whole request

// What a consumer needs to know about a block besides its K/V.
struct BlockInfo {
    int id;        // physical block
    int r;         // request (-1: no more blocks)
    int row;       // the request's packed row (query and output)
    int n_keys;    // ctx + 1
    uint32_t posf; // block index within the request | segment flags
};

struct __align__(1024) DecodeSmem {
    uint8_t kv[kDecStages][2][2][kHalfTile];   // [stage][K|V][dim half][row 16 h + token], 128-byte swizzle
    BlockInfo own[kIdCap];                      // the CTA's own part
    BlockInfo chunk[2][kMaxChunk];              // chunks taken from the pool (double-buffered)
    BlockInfo meta[kDecStages];                 // block in each stage
    int piece[kDecStages];
    int chunk_n[2], chunk_piece[2];             // blocks (0: the pool is empty) and piece of each chunk buffer
    int32_t page_off[kPageOffCap + 1];           // the step's block offsets, when they fit
    int stop;                                   // the producer asks the scheduler to leave
    uint64_t policy;
    uint64_t full[kDecStages], empty[kDecStages];
    uint64_t req;                               // producer -> scheduler: claim the next chunk
    uint64_t rdy[2];                            // scheduler -> producer: chunk buffer filled
};

static_assert(sizeof(DecodeSmem) + 1024 <= 227 * 1024, "decode CTA shared memory exceeds the per-CTA limit");

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

// How the P blocks are cut: G ranges of pp pieces each, the own part (piece 0 of a
// range) and pp - 1 chunks of its tail.  pp is the same for every range (so pieces
// number densely) and at most kMaxDecodeCtas / G (so r + piece stays inside the
// workspace's num_reqs + kMaxDecodeCtas partial slots).
struct Layout {
    int P, G, pp;
};

__device__ __forceinline__ Layout make_layout(int P, int G) {
    Layout L{P, G, 1};
    const int n_min = P / G;   // the shortest range
    const int n_ch = min(min(kMaxPieces, kMaxDecodeCtas / G) - 1, n_min * kTailPercent / 100 / kChunkTarget);
    if (n_ch >= 1) L.pp = 1 + n_ch;
    return L;
}

// Tail of a range of n blocks (0 when pp == 1).  Its n_ch = pp - 1 chunks shrink
// linearly: chunk k (0-based) gets a share n_ch - k of n_ch (n_ch + 1) / 2, so the last
// chunks handed out are the smallest and the CTAs that take them finish close together.
// The tail holds at least n_ch (n_ch + 1) / 2 blocks (so that no chunk is empty: make_layout
// keeps kChunkTarget n_ch <= n / 5 and n_ch <= 7) and at most 16 pp (so that the first, largest chunk
// has at most 2 tail / pp <= kMaxChunk blocks).
__device__ __forceinline__ int tail_blocks(const Layout& L, int n) {
    return L.pp > 1 ? min(n * kTailPercent / 100, 16 * L.pp) : 0;
}

// First block of chunk k of a tail, relative to the tail's start (k = n_ch: the tail's size).
__device__ __forceinline__ int chunk_start(int tail, int n_ch, int k) {
    const int sk = k * n_ch - k * (k - 1) / 2, total = n_ch * (n_ch + 1) / 2;
    return tail * sk / total;
}

// Global blocks [s, e) of piece pi.
__device__ __forceinline__ void piece_bounds(const Layout& L, int pi, int& s, int& e) {
    const int c = pi / L.pp, j = pi % L.pp;
    int lo, hi;
    cta_range(L.P, c, L.G, lo, hi);
    const int tail = tail_blocks(L, hi - lo), mid = hi - tail;
    if (j == 0) {
        s = lo;
        e = mid;
        return;
    }
    const int n_ch = L.pp - 1;
    s = mid + chunk_start(tail, n_ch, j - 1);
    e = mid + chunk_start(tail, n_ch, j);
}

// The piece holding global block x.
__device__ __forceinline__ int piece_of(const Layout& L, int x) {
    const int c = owner_cta(x, L.P, L.G);
    int lo, hi;
    cta_range(L.P, c, L.G, lo, hi);
    const int tail = tail_blocks(L, hi - lo), mid = hi - tail;
    if (x < mid) return c * L.pp;
    const int n_ch = L.pp - 1;
    int k = 0;
    while (k + 1 < n_ch && chunk_start(tail, n_ch, k + 1) <= x - mid) ++k;
    return c * L.pp + 1 + k;
}

// The largest r in [r_lo, num_reqs) with page_off[r] <= x (page_off[r_lo] <= x): the
// request that owns global block x (requests without decode blocks have empty ranges).
__device__ __forceinline__ int request_of(const int32_t* page_off, int num_reqs, int r_lo, int x) {
    int a = r_lo, step = 1;
    while (a + step < num_reqs && page_off[a + step] <= x) {
        a += step;
        step <<= 1;
    }
    int b = min(a + step - 1, num_reqs - 1);
    while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (page_off[mid] <= x) a = mid;
        else b = mid - 1;
    }
    return a;
}

// Everything a consumer needs about global block x of request r, in piece [s, e).
__device__ __forceinline__ BlockInfo block_info(int x, int r, int s, int e, const int32_t* page_off,
                                                const int32_t* tables, int max_blocks, int num_blocks,
                                                const int32_t* cu, const int32_t* ctx, uint32_t* err) {
    BlockInfo b;
    const int a0 = page_off[r], a1 = page_off[r + 1];
    const int pos = x - a0;
    int id = tables[(size_t)r * max_blocks + pos];
    if ((unsigned)id >= (unsigned)num_blocks) {
        raise_error(err, kErrBadBlock);
        id = 0;
    }
    b.id = id;
    b.r = r;
    b.row = cu[r];
    b.n_keys = ctx[r] + 1;
    b.posf = (uint32_t)pos | ((x == s || x == a0) ? kFirst : 0u) | ((x == e - 1 || x == a1 - 1) ? kLast : 0u) |
             ((a0 >= s && a1 <= e) ? kWhole : 0u);
    return b;
}

struct DecodeArgs {
    const __nv_bfloat16* q;
    __nv_bfloat16* out;
    const int32_t* cu;
    const int32_t* ctx;
    const int32_t* tables;
    int max_blocks;
    int num_blocks;
    const int32_t* page_off;
    int num_reqs;
    int wave;
    int32_t* counters;   // [2]: decode CTAs wanted, [4]: chunks taken
    float* part_acc;
    float2* part_ml;
    float scale_log2;
    uint32_t* err;
};

// The scheduler warp: on each request of the producer, claims the next chunk from the
// pool (one global counter) and describes its blocks into chunk buffer i % 2 (the
// producer has finished issuing the chunk that buffer held before).  Leaves after handing
// over an empty chunk, or when the producer asks it to.
__device__ __forceinline__ void schedule(DecodeSmem& S, const DecodeArgs& a, const Layout& L, int lane) {
    const int n_chunks = L.G * (L.pp - 1);
    for (int i = 0;; ++i) {
        if (!warp_wait(&S.req, (uint32_t)(i & 1))) {
            if (lane == 0) raise_error(a.err, kErrTimeout);
            return;
        }
        if (*(volatile int*)&S.stop) return;
        const int buf = i & 1;
        int kk = 0;
        if (lane == 0) kk = atomicAdd(&a.counters[4], 1);
        kk = __shfl_sync(0xffffffffu, kk, 0);
        int n = 0, piece = 0;
        if (kk < n_chunks) {
            piece = (kk % L.G) * L.pp + 1 + kk / L.G;
            int s, e;
            piece_bounds(L, piece, s, e);
            // request of block s: a 32-way search over page_off, then each lane its own block
            int ra = 0, rb = a.num_reqs - 1;
            while (ra < rb) {
                const int step = (rb - ra + 32) / 32;
                const int idx = ra + lane * step;
                const unsigned m = __ballot_sync(0xffffffffu, idx <= rb && a.page_off[idx] <= s);
                ra += (31 - __clz(m)) * step;
                rb = min(rb, ra + step - 1);
            }
            n = min(e - s, kMaxChunk);
            if (lane < n) {
                const int x = s + lane;
                const int r = request_of(a.page_off, a.num_reqs, ra, x);
                S.chunk[buf][lane] =
                    block_info(x, r, s, e, a.page_off, a.tables, a.max_blocks, a.num_blocks, a.cu, a.ctx, a.err);
            }
        }
        __syncwarp();
        if (lane == 0) {
            S.chunk_n[buf] = n;
            S.chunk_piece[buf] = piece;
            mbar_arrive(&S.rdy[buf]);   // release: the lanes' descriptions are ordered by the __syncwarp
        }
        if (n == 0) return;
    }
}

// The producer warp: issues the CTA's own part, then the chunks the scheduler claims,
// one block per free stage; ends with a stage that carries r = -1.  It asks for the next
// chunk kClaimLead blocks before the end of the own part and at the start of each chunk,
// so that the claim and its table lookups run while earlier blocks stream.
__device__ __forceinline__ void produce(DecodeSmem& S, const DecodeArgs& a, const CUtensorMap* tk,
                                        const CUtensorMap* tv, const Layout& L, int n_own, int cta, int lane) {
    int k = 0;   // blocks issued
    bool ok = true;
    // Whole warp, in step: wait for stage k % kDecStages to be free; one elected lane
    // describes the block and issues its copies (operands the same in every lane: a lone
    // lane running this loop issued its instructions far more slowly).
    const bool leader = elect_one();
    auto issue = [&](const BlockInfo& b, int piece) -> bool {
        const int st = k % kDecStages;
        if (!warp_wait(&S.empty[st], ((k / kDecStages) & 1) ^ 1)) return false;
        const int y = b.id * kBlockRows;
        const uint32_t bar = smem_u32(&S.full[st]);
        const uint32_t d = smem_u32(S.kv[st][0][0]);
        if (leader) {
            S.meta[st] = b;
            S.piece[st] = piece;
            mbar_arrive_expect_tx(&S.full[st], kStageBytes);
            tma_load_2d_hint(d, tk, 0, y, bar, S.policy);
            tma_load_2d_hint(d + kHalfTile, tk, 64, y, bar, S.policy);
            tma_load_2d_hint(d + 2 * kHalfTile, tv, 0, y, bar, S.policy);
            tma_load_2d_hint(d + 3 * kHalfTile, tv, 64, y, bar, S.policy);
        }
        __syncwarp();
        return true;
    };
    int n_req = 0, n_got = 0;   // chunks asked for, chunks received
    auto request = [&]() {
        if (lane == 0) mbar_arrive(&S.req);
        ++n_req;
    };
    // whole warp: the next chunk's blocks (0: the pool is empty, -1: the wait ran out)
    auto receive = [&](int& buf, int& piece) -> int {
        buf = n_got & 1;
        const bool w = warp_wait(&S.rdy[buf], (uint32_t)((n_got >> 1) & 1));
        ++n_got;
        if (!w) return -1;
        piece = S.chunk_piece[buf];
        return S.chunk_n[buf];
    };

    const bool pool = L.pp > 1;
    const int own_piece = cta * L.pp;
    const int claim_at = max(0, n_own - kClaimLead);
    // The first blocks (described by this warp) go out before the rest of the own part is
    // described by the other warps; then the CTA meets once.
    const int q_pre = min(kDecStages, n_own);
    int q = 0;
    for (; q < q_pre && ok; ++q) {
        if (q == claim_at && pool) request();
        ok = issue(S.own[q], own_piece);
        ++k;
    }
    __syncthreads();   // the own part is described; every warp sees the barriers initialised
    for (; q < n_own && ok; ++q) {
        if (q == claim_at && pool) request();
        ok = issue(S.own[q], own_piece);
        ++k;
    }
    int n = 0, buf = 0, piece = 0;
    bool sched_done = !pool;   // the scheduler has handed over an empty chunk and left
    if (ok && pool) n = receive(buf, piece);
    while (ok && n > 0) {
        // the chunk after this one (into the other buffer) is claimed kClaimLead blocks
        // before this one is all issued
        const int req_at = max(0, n - kClaimLead);
        for (int j = 0; j < n && ok; ++j) {
            if (j == req_at) request();
            ok = issue(S.chunk[buf][j], piece);
            ++k;
        }
        if (ok) n = receive(buf, piece);
    }
    if (n < 0) ok = false;
    if (ok && pool) sched_done = true;   // the loop ended on n == 0
    if (lane == 0) {
        if (!sched_done && n_req == n_got) {
            // stopped early (an error) with no claim outstanding: let the scheduler go
            *(volatile int*)&S.stop = 1;
            mbar_arrive(&S.req);
        }
        bool ended = false;
        if (ok) {
            // no more blocks: a stage without a copy, r = -1
            const int st = k % kDecStages;
            if (mbar_wait(&S.empty[st], ((k / kDecStages) & 1) ^ 1)) {
                S.meta[st].r = -1;
                mbar_arrive(&S.full[st]);
                ended = true;
            }
        }
        if (!ok || !ended) raise_error(a.err, kErrTimeout);
        // The CTA must not retire while a copy still targets its shared memory: wait for
        // the last blocks issued into each stage (the stage of the end marker was seen
        // consumed already).
        for (int j = max(0, k - kDecStages); j < k; ++j) {
            if (ended && j % kDecStages == k % kDecStages) continue;
            if (!mbar_wait(&S.full[j % kDecStages], (uint32_t)((j / kDecStages) & 1))) raise_error(a.err, kErrTimeout);
        }
    }
}

// A consumer warp (KV head h): every block of the CTA's sequence, in stage order.
__device__ __forceinline__ void consume(DecodeSmem& S, const DecodeArgs& a, const Layout& L, int h, int lane) {
    // Fragment coordinates (PTX mma.m16n8k16 layouts): lane = 4 g + t.  A fragment rows
    // are tokens (S^T) or dims (O^T); B columns and C columns are the query heads, of
    // which columns 0..3 are real (lanes with t < 2 hold them in C).
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
    uint32_t qb[8][2];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // heads 2t, 2t + 1
    float o[8][4];
    for (int k = 0;; ++k) {
        const int stage = k % kDecStages;
        if (!warp_wait(&S.full[stage], (uint32_t)((k / kDecStages) & 1))) {
            if (lane == 0) raise_error(a.err, kErrTimeout);
            return;
        }
        const BlockInfo b = S.meta[stage];
        if (b.r < 0) return;
        const int piece = S.piece[stage];
        if (b.posf & kFirst) {
            // Q^T as the B operand of S^T = K Q^T: k-step s covers dims 16 s .. 16 s + 15;
            // lane (g, t) holds head g's dims 16 s + 2 t, +1 and 16 s + 2 t + 8, +9 (zero
            // for g >= 4)
            const uint32_t* qw = reinterpret_cast<const uint32_t*>(a.q + (size_t)b.row * kQRowElems +
                                                                    (h * kGroup + (g & 3)) * kHeadDim);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                qb[s][0] = g < kGroup ? __ldg(qw + 8 * s + t) : 0u;
                qb[s][1] = g < kGroup ? __ldg(qw + 8 * s + 4 + t) : 0u;
            }
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        }
        const uint32_t kb = ring0 + stage * kStageBytes, vb = kb + 2 * kHalfTile;
        const int n_valid = b.n_keys - (int)(b.posf & kPosMask) * kBlockSize;   // >= 1; < 16 only in a last block
        // All of this warp's reads of the stage first (K and V fragments into registers),
        // then the stage is released, so the refill starts before the arithmetic.
        uint32_t ka[8][4], va[8][4];
#pragma unroll
        for (int s = 0; s < 8; ++s) ldsm_x4(kb + (s >> 2) * kHalfTile + k_off[s & 3], ka[s]);
#pragma unroll
        for (int i = 0; i < 8; ++i) ldsm_x4_t(vb + (i >> 2) * kHalfTile + v_off[i & 3], va[i]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[stage]);
        if (n_valid < kBlockSize) {
            // tokens past the end of the request: zero their V values (stale bytes could
            // hold NaN, and 0 x NaN is NaN).  V^T fragment registers 0, 1 hold tokens 2t,
            // 2t + 1; registers 2, 3 tokens 2t + 8, 2t + 9.
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
        for (int j = 0; j < 4; ++j) x[j] = (sa[j] + sb[j]) * a.scale_log2;
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

        if (!(b.posf & kLast)) continue;
        // ------------------------------------------------ end of a segment
        float s0 = l0, s1 = l1;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, off);
            s1 += __shfl_xor_sync(0xffffffffu, s1, off);
        }
        if (b.posf & kWhole) {
            // O = O^T / l, transposed back so that lane (g, t) holds dims 16 i + 2t, +1
            // and 16 i + 8 + 2t, +1 of head g
            const float i0 = s0 > 0.f ? 1.f / s0 : 0.f, i1 = s1 > 0.f ? 1.f / s1 : 0.f;
            uint32_t* orow = reinterpret_cast<uint32_t*>(a.out + (size_t)b.row * kQRowElems +
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
            continue;
        }
        // Split row: this piece's partial for the warp's 4 query heads, merged with the
        // row's other pieces by the combine kernel that follows the step's attention
        // kernels (so no consumer waits on global memory here).
        const size_t slot = (size_t)b.r + piece;
        if (t < 2) {
            float* pa = a.part_acc + (slot * kNumQHeads + h * kGroup + 2 * t) * kHeadDim;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                pa[16 * i + g] = o[i][0];
                pa[kHeadDim + 16 * i + g] = o[i][1];
                pa[16 * i + 8 + g] = o[i][2];
                pa[kHeadDim + 16 * i + 8 + g] = o[i][3];
            }
            if (g == 0) {
                a.part_ml[slot * kNumQHeads + h * kGroup + 2 * t] = make_float2(m0, s0);
                a.part_ml[slot * kNumQHeads + h * kGroup + 2 * t + 1] = make_float2(m1, s1);
            }
        }
    }
}

// The body of one decode CTA: CTA `cta` of a launch of `grid` CTAs shares out the step's
// decode blocks (the decode kernel runs it with its block index and grid size; the mixed
// step kernel with the decode CTA index its work ticket names).  Uses threads 0 .. 319 (10
// warps); any further threads of the CTA meet its one block-wide barrier and leave.
__device__ __forceinline__ void decode_cta(const CUtensorMap& tmap_k, const CUtensorMap& tmap_v, const DecodeArgs& a,
                                           DecodeSmem& S, int cta, int grid) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    grid_dep_wait();     // block offsets, cache contents
    grid_dep_launch();
    // the block offsets go to shared memory (one coalesced pass) when they fit, so that
    // every search below runs there
    DecodeArgs b = a;
    const int want = a.counters[2];   // the decode's share of the SMs (loaded alongside the offsets)
    if (a.num_reqs <= kPageOffCap) {
        for (int k = threadIdx.x; k <= a.num_reqs; k += blockDim.x) S.page_off[k] = a.page_off[k];
        __syncthreads();
        b.page_off = S.page_off;
    }
    const int32_t* po = b.page_off;
    const int P = po[a.num_reqs];
    if (P <= 0) return;
    // SMs left to this step's prefill tiles run them meanwhile (unless the launch is too
    // small for the narrower waves that would need)
    int G = decode_ctas_used(P, max(1, min(a.wave, want)), grid);
    if (G == 0) G = decode_ctas_used(P, a.wave, grid);
    if (G == 0) {
        // the launch has too few CTAs for this many blocks (the host sizes it from an
        // upper bound, so this means inconsistent metadata)
        if (cta == 0 && threadIdx.x == 0) raise_error(a.err, kErrBadMeta);
        return;
    }
    if ((int)cta >= G) return;
    const Layout L = make_layout(P, G);
    int lo, mid;
    piece_bounds(L, (int)cta * L.pp, lo, mid);   // the own part
    const int n_own = mid - lo;   // >= 1 and <= kIdCap by construction of G
    if (n_own < 1 || n_own > kIdCap) {
        if (threadIdx.x == 0) raise_error(a.err, kErrBadMeta);
        return;
    }

    // ids, requests and positions of every block of the own part (requests found by
    // searches between those of its first and its last block): the producer warp describes
    // the first 32 and starts copying at once, the other warps describe the rest
    const int r_first = request_of(po, a.num_reqs, 0, lo);
    const int r_last = request_of(po, a.num_reqs, r_first, mid - 1);
    auto describe = [&](int x) {
        int ra = r_first, rb = r_last;   // largest r with page_off[r] <= x
        while (ra < rb) {
            const int m = (ra + rb + 1) >> 1;
            if (po[m] <= x) ra = m;
            else rb = m - 1;
        }
        S.own[x - lo] = block_info(x, ra, lo, mid, po, a.tables, a.max_blocks, a.num_blocks, a.cu, a.ctx, a.err);
    };
    if (warp == kProducerWarp) {
        if (lane == 0) {
            for (int s = 0; s < kDecStages; ++s) {
                mbar_init(&S.full[s], 1);
                mbar_init(&S.empty[s], kConsumerWarps);
            }
            mbar_init(&S.req, 1);
            mbar_init(&S.rdy[0], 1);
            mbar_init(&S.rdy[1], 1);
            S.stop = 0;
            S.policy = policy_evict_first();
            fence_barrier_init();
        }
        if (lo + lane < mid) describe(lo + lane);
        __syncwarp();
        produce(S, b, &tmap_k, &tmap_v, L, n_own, cta, lane);   // meets the other warps' __syncthreads
        return;
    }
    const int t = warp < kProducerWarp ? (int)threadIdx.x : (int)threadIdx.x - 32;   // among the other warps
    if (t < kDecThreads - 32)
        for (int x = lo + 32 + t; x < mid; x += kDecThreads - 32) describe(x);
    __syncthreads();
    if (warp == kSchedulerWarp) {
        if (L.pp > 1) schedule(S, b, L, lane);
    } else if (warp < kConsumerWarps) {
        consume(S, b, L, warp, lane);
    }}

// CTAs that run at once: one per SM, or fewer when the pool asks for fewer.
inline int decode_wave(const StepArgs& a) {
    int w = a.num_sms > 0 ? a.num_sms : 1;
    if (w > kMaxDecodeCtas) w = kMaxDecodeCtas;
    if (a.decode_ctas > 0 && a.decode_ctas < w) w = a.decode_ctas;
    return w;
}

// Launch size: whole waves, enough that no CTA's share exceeds kIdCap blocks for the
// largest decode work these arguments allow (every request a decode row at the maximum
// context); capped at kMaxDecodeCtas (the kernel flags a step that would need more).
inline int decode_grid(const StepArgs& a, int wave) {
    const long long per_req = ((long long)a.max_context_len + 1 + kBlockSize - 1) / kBlockSize;
    const long long p_upper = per_req * (long long)a.num_reqs;
    const long long per_launch_wave = (long long)wave * kIdCap;
    long long waves = (p_upper + per_launch_wave - 1) / per_launch_wave;
    if (waves < 1) waves = 1;
    const long long max_waves = kMaxDecodeCtas / wave;
    if (waves > max_waves) waves = max_waves > 0 ? max_waves : 1;
    return (int)(waves * wave);
}

// The decode kernel's arguments for one step.
inline DecodeArgs make_decode_args(const StepArgs& a) {
    const StepLayout& L = a.lay;
    DecodeArgs d;
    d.q = static_cast<const __nv_bfloat16*>(a.q);
    d.out = static_cast<__nv_bfloat16*>(a.out);
    d.cu = a.cu_seqlens_q;
    d.ctx = a.context_lens;
    d.tables = a.block_tables;
    d.max_blocks = a.max_blocks_per_seq;
    d.num_blocks = a.num_blocks;
    d.page_off = reinterpret_cast<const int32_t*>(a.ws + L.page_off_off);
    d.num_reqs = a.num_reqs;
    d.wave = decode_wave(a);
    d.counters = reinterpret_cast<int32_t*>(a.ws + L.counters_off);
    d.part_acc = reinterpret_cast<float*>(a.ws + L.part_acc_off);
    d.part_ml = reinterpret_cast<float2*>(a.ws + L.part_ml_off);
    d.scale_log2 = a.softmax_scale * 1.4426950408889634f;
    d.err = a.err;
    return d;
}

}  // namespace
}  // namespace kvp
