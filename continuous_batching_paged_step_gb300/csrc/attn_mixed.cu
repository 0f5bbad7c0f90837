// Mixed step kernel: one persistent launch for a step's decode rows and prefill tiles.
//
// Page "Continuous Batching" (k4i.top), section "把 prefill 和 decode 打包在一起", and
// page "11.2 连续批处理与 PagedAttention", section 11.2.2 (Figure 11-3): a step's prefill
// chunks and decode rows are one packed pass.  This kernel gives that pass one grid of
// the decode launch's size (whole waves of one CTA per SM).  Each CTA, once the step's
// metadata kernel is complete, takes a work ticket from a device counter:
//   tickets [0, D): decode CTA t of D (the decode kernel's CTA body: its block range with
//     the 20 % tail handed out as chunks through a second counter; tickets beyond the
//     share of SMs the metadata kernel gives the decode have no range);
// and then, whatever its ticket, takes prefill work items (tile, KV head) from a third
// counter, in the metadata kernel's longest-first order, until none are left (the prefill
// kernel's CTA body, its rings, barriers and TMEM carried from item to item).  CTAs take
// tickets in the order they start, so the decode ranges start first, spread over the GPU;
// the CTAs without a range start on prefill items at once, and every decode CTA joins them
// when its range is done, so the prefill tail runs on every SM.  Split decode rows are
// merged by the combine kernel after this one.
#include "attn_decode.cuh"
#include "attn_prefill.cuh"

namespace kvp {

namespace {

constexpr int kMixedThreads = kPreThreads;   // 12 warps (the decode CTA body uses 10)
constexpr size_t kMixedSmemBytes =
    (sizeof(DecodeSmem) > sizeof(PrefillSmem) ? sizeof(DecodeSmem) : sizeof(PrefillSmem)) + 1024;
static_assert(kMixedSmemBytes <= 227 * 1024, "mixed step CTA shared memory exceeds the per-CTA limit");
static_assert(kDecThreads <= kMixedThreads, "the decode CTA body needs at most the mixed CTA's threads");

struct MixedArgs {
    DecodeArgs d;
    PrefillArgs p;
    int decode_slots;   // tickets of decode CTAs (the decode launch's size)
    int32_t* ticket;    // work ticket counter (zeroed by the metadata kernel)
};

__global__ void __launch_bounds__(kMixedThreads, 1)
    mixed_step_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_k_blk,
                      const __grid_constant__ CUtensorMap tmap_v_blk, const MixedArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ int s_ticket;
    grid_dep_wait();   // the metadata kernel: work lists, the zeroed counters, the appended K/V
    if (threadIdx.x == 0) s_ticket = atomicAdd(a.ticket, 1);
    __syncthreads();
    const int t = s_ticket;
    if (t < a.decode_slots) {
        decode_cta(tmap_k_blk, tmap_v_blk, a.d, *reinterpret_cast<DecodeSmem*>(base), t, a.decode_slots);
        __syncthreads();   // every warp is done with the decode body's shared memory
    }
    grid_dep_launch();
    // prefill items until none are left, the first claimed before any set-up
    __shared__ int s_first;
    if (threadIdx.x == 0) {
        const int k = atomicAdd(a.p.next_item, 1);
        s_first = k < __ldcg(&a.p.counters[1]) * kNumKvHeads ? k : -1;
    }
    __syncthreads();
    if (s_first >= 0)
        prefill_cta(tmap_q, tmap_k, tmap_v, a.p, *reinterpret_cast<PrefillSmem*>(base), s_first, a.p.next_item);
}

}  // namespace

cudaError_t launch_mixed(const StepArgs& a, const CUtensorMap* tmap_q, const CUtensorMap* tmap_k,
                         const CUtensorMap* tmap_v, const CUtensorMap* tmap_k_blk, const CUtensorMap* tmap_v_blk,
                         cudaStream_t stream) {
    MixedArgs m;
    m.d = make_decode_args(a);
    m.decode_slots = decode_grid(a, decode_wave(a));
    const bool prefill = a.max_q_len >= 2 && a.lay.max_prefill_tiles > 0;
    m.p = make_prefill_args(a);
    int32_t* counters = reinterpret_cast<int32_t*>(a.ws + a.lay.counters_off);
    m.ticket = counters + 5;
    // the decode launch's size; at least as many CTAs as prefill items run at once
    long long grid = m.decode_slots;
    if (prefill) {
        const long long items = (long long)a.lay.max_prefill_tiles * kNumKvHeads;
        const long long want = items < a.num_sms ? items : a.num_sms;
        if (grid < want) grid = want;
    }
    return launch_pdl(mixed_step_kernel, dim3((unsigned)grid), dim3(kMixedThreads), kMixedSmemBytes, stream, *tmap_q,
                      *tmap_k, *tmap_v, *tmap_k_blk, *tmap_v_blk, m);
}

cudaError_t configure_mixed_kernel() {
    return cudaFuncSetAttribute(mixed_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMixedSmemBytes);
}

}  // namespace kvp
