// Decode kernel and split-KV combine kernel, and their launches (the decode device code is
// in attn_decode.cuh).
#include "attn_decode.cuh"

namespace kvp {

namespace {

__global__ void __launch_bounds__(kDecThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    DecodeSmem& S =
        *reinterpret_cast<DecodeSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    decode_cta(tmap_k, tmap_v, a, S, (int)blockIdx.x, (int)gridDim.x);
}

constexpr int kCombineStage = 12;                     // pieces staged in shared memory at once
constexpr int kCombineStageWide = 20;                 // ... when there are few rows (one round for long rows)
// query heads of one combine CTA when a row's merge is split over `parts` CTAs, and that
// CTA's share of one piece: accumulators (head x 128 fp32) and (m, l) per head
__host__ __device__ constexpr int combine_heads(int parts) { return kNumQHeads / parts; }
__host__ __device__ constexpr int combine_acc_bytes(int parts) { return combine_heads(parts) * kHeadDim * 4; }
__host__ __device__ constexpr int combine_ml_bytes(int parts) { return combine_heads(parts) * 8; }

constexpr int kCombineRowsPerRound = 32;   // rows a CTA plans at once

// Shared memory of a combine CTA staging `stage` pieces: this header, then the pieces'
// accumulators and their (m, l) (this CTA's heads of them).
struct CombineSmem {
    int4 job[kCombineRowsPerRound];   // {request, row, first piece, last piece} of the rows to merge
    int n_job;
    uint64_t full;
};

__host__ __device__ constexpr size_t combine_smem_bytes(int stage, int parts) {
    return ((sizeof(CombineSmem) + 127) & ~size_t(127)) +
           (size_t)stage * (combine_acc_bytes(parts) + combine_ml_bytes(parts)) + 128;
}

// Split-KV combine: every decode row whose blocks the decode kernel cut into several
// pieces gets O = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p over its pieces
// (M = max_p m_p), merged online piece by piece.  kParts CTAs per row (32 / kParts
// query heads each, one warp per head, lane l holding dims 4l .. 4l + 3); a CTA stages up
// to `stage` pieces' partials at once in shared memory with bulk copies, so a row costs
// about one round trip to memory.  Rows held by one piece were finished in place.  Launched after
// the step's attention kernels, as a programmatic dependent: before its wait it works out
// its row's pieces from the metadata kernel's outputs (complete before the decode kernel
// let its dependents launch) and the decode launch's size; after the wait (for the decode
// grid; the prefill grid, when there is one, completes only after it) only the copies and
// the merge remain.
template <int kParts>
__global__ void __launch_bounds__(kNumQHeads / kParts * 32) combine_kernel(const int32_t* __restrict__ page_off, int num_reqs,
                                                                   const int32_t* __restrict__ cu,
                                                                   const int32_t* __restrict__ counters,
                                                                   int decode_wave, int decode_grid,
                                                                   const float* __restrict__ part_acc,
                                                                   const float2* __restrict__ part_ml,
                                                                   __nv_bfloat16* __restrict__ out,
                                                                   uint32_t* __restrict__ err, int stage) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    CombineSmem& S = *reinterpret_cast<CombineSmem*>(base);
    constexpr int kCombineHeads = combine_heads(kParts);
    constexpr int kCombineAccBytes = combine_acc_bytes(kParts), kCombineMlBytes = combine_ml_bytes(kParts);
    float* s_acc = reinterpret_cast<float*>(base + ((sizeof(CombineSmem) + 127) & ~size_t(127)));   // [stage][heads][128]
    float2* s_ml = reinterpret_cast<float2*>(s_acc + (size_t)stage * kCombineHeads * kHeadDim);      // [stage][heads]
    const int part = (int)(blockIdx.x % kParts);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int head = part * kCombineHeads + warp;
    uint32_t phase = 0;
    if (threadIdx.x == 0) {
        mbar_init(&S.full, 1);
        fence_barrier_init();
    }
    // This group of kParts CTAs takes rows blockIdx.x / kParts + k * stride; it plans up to
    // kCombineRowsPerRound of them at once (one thread each), then merges those to merge.
    const int stride = (int)(gridDim.x / kParts);
    for (int r0 = (int)(blockIdx.x / kParts); r0 < num_reqs; r0 += kCombineRowsPerRound * stride) {
        if (threadIdx.x == 0) S.n_job = 0;
        __syncthreads();
        const int r = r0 + (int)threadIdx.x * stride;
        if (threadIdx.x < kCombineRowsPerRound && r < num_reqs) {
            // every load at once, then the arithmetic
            const int P = page_off[num_reqs], want = counters[2];
            const int a0 = page_off[r], a1 = page_off[r + 1], row = cu[r];
            int G = 0;   // the decode kernel's CTA count, as it works it out
            if (P > 0) {
                G = decode_ctas_used(P, max(1, min(decode_wave, want)), decode_grid);
                if (G == 0) G = decode_ctas_used(P, decode_wave, decode_grid);
            }
            if (G > 0 && a1 > a0) {   // a decode row
                const Layout L = make_layout(P, G);
                const int p0 = piece_of(L, a0), p1 = piece_of(L, a1 - 1);
                if (p0 != p1) S.job[atomicAdd(&S.n_job, 1)] = make_int4(r, row, p0, p1);   // else finished in place
            }
        }
        __syncthreads();
        const int n_job = S.n_job;
        if (n_job > 0) grid_dep_wait();   // the decode kernel's partials
        for (int ji = 0; ji < n_job; ++ji) {
            const int4 job = S.job[ji];
            float M = -INFINITY, L = 0.f;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int b = job.z; b <= job.w; b += stage) {
                const int nb = min(stage, job.w - b + 1);
                if (threadIdx.x == 0) {
                    fence_proxy_async_smem();   // earlier reads of the stage before the copies' writes
                    mbar_arrive_expect_tx(&S.full, (uint32_t)(nb * (kCombineAccBytes + kCombineMlBytes)));
                    const uint64_t pol = policy_evict_first();
                    for (int j = 0; j < nb; ++j) {
                        const size_t slot = (size_t)job.x + b + j;
                        bulk_load(s_acc + (size_t)j * kCombineHeads * kHeadDim,
                                  part_acc + (slot * kNumQHeads + part * kCombineHeads) * kHeadDim, kCombineAccBytes,
                                  &S.full, pol);
                        bulk_load(s_ml + j * kCombineHeads, part_ml + slot * kNumQHeads + part * kCombineHeads,
                                  kCombineMlBytes, &S.full,
                                  pol);
                    }
                }
                // thread 0's warp waits on the barrier together, once the copies are out (lanes
                // of that warp that waited on it while thread 0 was held up elsewhere went on
                // before the copies had landed)
                __syncwarp();
                if (!mbar_wait(&S.full, phase)) {
                    // the copies did not land within the wait limit; they target this CTA's shared
                    // memory, so give them another bounded wait before leaving
                    if (lane == 0) raise_error(err, kErrTimeout);
                    if (threadIdx.x == 0) mbar_wait(&S.full, phase);
                    return;
                }
                phase ^= 1;
                for (int j = 0; j < nb; ++j) {
                    const float2 ml = s_ml[j * kCombineHeads + warp];
                    const float4 v = reinterpret_cast<const float4*>(s_acc + ((size_t)j * kCombineHeads + warp) * kHeadDim)[lane];
                    const float Mn = fmaxf(M, ml.x);   // finite: every piece holds a key
                    const float c = fast_exp2(M - Mn), w = fast_exp2(ml.x - Mn);
                    L = fmaf(L, c, ml.y * w);
                    o.x = fmaf(o.x, c, v.x * w);
                    o.y = fmaf(o.y, c, v.y * w);
                    o.z = fmaf(o.z, c, v.z * w);
                    o.w = fmaf(o.w, c, v.w * w);
                    M = Mn;
                }
                __syncthreads();   // the stage is free again
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
            uint2 wv;
            wv.x = pack_bf16x2(o.x * inv, o.y * inv);
            wv.y = pack_bf16x2(o.z * inv, o.w * inv);
            reinterpret_cast<uint2*>(out + (size_t)job.y * kQRowElems + head * kHeadDim)[lane] = wv;
        }
        __syncthreads();   // S.job and S.n_job are rewritten next round
    }
    // What follows in the stream (the next step's kernels: its metadata kernel resets the work
    // counters and rewrites the work lists) starts only once the step's attention kernels have
    // completed; a CTA with no rows to merge has not waited for them above.
    grid_dep_wait();
    grid_dep_launch();
}

}  // namespace

cudaError_t launch_decode(const StepArgs& a, const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                          cudaStream_t stream) {
    const size_t smem = sizeof(DecodeSmem) + 1024;
    return launch_pdl(decode_kernel, dim3(decode_grid(a, decode_wave(a))), dim3(kDecThreads), smem, stream, *tmap_k,
                      *tmap_v, make_decode_args(a));
}

cudaError_t launch_combine(const StepArgs& a, cudaStream_t stream) {
    const StepLayout& L = a.lay;
    const int wave = decode_wave(a);
    // No more CTAs than run at once, each group then taking several rows.  With few rows
    // (4 per row fit two to an SM) four CTAs of 8 heads share each row and stage 20 pieces
    // at once, so the longest rows of a mixed step cost one round trip of ~80 KiB per SM;
    // with at most as many rows as SM pairs, two CTAs of 16 heads per row, each with an SM
    // to itself; otherwise two such CTAs per SM stage 12 pieces each.  (Three CTAs per SM
    // staging 8 pieces each merged the 256-row decode step more slowly: its longest rows
    // took more rounds.)
    const long long sms = a.num_sms > 0 ? a.num_sms : 1;
    const bool quarter = 4LL * a.num_reqs <= 2 * sms;
    const bool wide = 2LL * a.num_reqs <= sms;
    const int parts = quarter ? 4 : 2;
    const int stage = (quarter || wide) ? kCombineStageWide : kCombineStage;
    long long grid = (long long)parts * a.num_reqs;
    const long long cap = quarter ? 2 * sms / 4 * 4 : wide ? sms / 2 * 2 : 2LL * sms;
    if (grid > cap) grid = cap;
    if (grid < parts) grid = parts;
    auto go = [&](auto kernel) {
        return launch_pdl(kernel, dim3((unsigned)grid), dim3(kNumQHeads / parts * 32), combine_smem_bytes(stage, parts),
                          stream, reinterpret_cast<const int32_t*>(a.ws + L.page_off_off), a.num_reqs, a.cu_seqlens_q,
                          reinterpret_cast<const int32_t*>(a.ws + L.counters_off), wave, decode_grid(a, wave),
                          reinterpret_cast<const float*>(a.ws + L.part_acc_off),
                          reinterpret_cast<const float2*>(a.ws + L.part_ml_off), static_cast<__nv_bfloat16*>(a.out),
                          a.err, stage);
    };
    return quarter ? go(combine_kernel<4>) : go(combine_kernel<2>);
}

cudaError_t configure_decode_kernel() {
    const cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)(sizeof(DecodeSmem) + 1024));
    if (e != cudaSuccess) return e;
    const cudaError_t e2 = cudaFuncSetAttribute(combine_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)combine_smem_bytes(kCombineStageWide, 2));
    if (e2 != cudaSuccess) return e2;
    return cudaFuncSetAttribute(combine_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)combine_smem_bytes(kCombineStageWide, 4));
}

}  // namespace kvp
