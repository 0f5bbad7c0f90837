// Prefill kernel and its launch (the prefill device code is in attn_prefill.cuh).
#include "attn_prefill.cuh"

namespace kvp {

namespace {

// Launched right after the decode kernel, as its programmatic dependent: CTAs start as
// soon as every decode CTA has passed its own wait for the step's metadata kernel (so the
// work list and the appended K/V are complete) and take the SMs the decode leaves free,
// at most one per SM; each takes work items from the step's counter until none are left,
// so CTAs that start late (on SMs the decode frees) still find work.  The grid finishes
// only after the decode grid has: its last CTA to leave waits for it.
__global__ void __launch_bounds__(kPreThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    PrefillSmem& S =
        *reinterpret_cast<PrefillSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ int s_first;
    grid_dep_launch();
    // the CTA's first item, claimed before any set-up: a CTA that finds none leaves at once
    if (threadIdx.x == 0) {
        const int k = atomicAdd(a.next_item, 1);
        s_first = k < __ldcg(&a.counters[1]) * kNumKvHeads ? k : -1;
    }
    __syncthreads();
    if (s_first >= 0) prefill_cta(tmap_q, tmap_k, tmap_v, a, S, s_first, a.next_item);
    __syncthreads();
    if (threadIdx.x == 0) {
        if (atomicAdd(a.done, 1) == (int)gridDim.x - 1) grid_dep_wait();
    }
}

}  // namespace

cudaError_t launch_prefill(const StepArgs& a, const CUtensorMap* tmap_q, const CUtensorMap* tmap_k,
                           const CUtensorMap* tmap_v, cudaStream_t stream) {
    const StepLayout& L = a.lay;
    if (L.max_prefill_tiles <= 0 || a.max_q_len < 2) return cudaSuccess;
    const PrefillArgs pa = make_prefill_args(a);
    const long long items = (long long)L.max_prefill_tiles * kNumKvHeads;
    const int grid = (int)(items < a.num_sms ? items : a.num_sms);
    const size_t smem = sizeof(PrefillSmem) + 1024;
    return launch_pdl(prefill_kernel, dim3(grid), dim3(kPreThreads), smem, stream, *tmap_q, *tmap_k, *tmap_v, pa);
}

cudaError_t configure_prefill_kernel() {
    return cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(sizeof(PrefillSmem) + 1024));
}

}  // namespace kvp
