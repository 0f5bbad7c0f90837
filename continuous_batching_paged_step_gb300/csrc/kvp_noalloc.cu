// paged_attention_step_noalloc: the attention step for callers that cannot allocate
// device memory.
//
// paged_attention_step takes its scratch (work lists and split-KV partial results) from
// a caller-provided workspace.  Some callers cannot provide one at step time: an engine
// that has given all free device memory to its KV pool and forbids later allocations,
// or a host that must not call cudaMalloc / cudaFree from its serving loop because they
// may synchronise the device.  This entry point uses instead a fixed scratch array that
// lives in this library's device code (a file-scope __device__ array), so a call
// allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
//
// Costs and limits of that choice:
// * Every GPU that loads the library holds the array (kNoAllocScratchBytes) until the
//   process exits, whether or not this entry point is ever called.
// * All calls share the one array: two calls whose kernels overlap on the GPU (on
//   different streams, or from different threads) race on it and corrupt each other.
//   Calls in the same stream are ordered and safe.
// * Nothing in the array needs to start at zero: each call writes every scratch value
//   it later reads.
// * A step whose scratch would not fit is rejected with KVP_E_WORKSPACE before anything
//   is launched.
// * The array's device address is looked up once per device (cudaGetSymbolAddress, with
//   that device current) on the first call made with that device current; make that
//   first call before any stream capture begins.
#include <cuda_runtime.h>

#include <mutex>

#include "kvpaged.h"
#include "kvp_launch.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on `dev` (the current device), looked up once.
void* scratch_address(int dev) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" KVP_API size_t paged_attention_noalloc_capacity(void) { return kNoAllocScratchBytes; }

extern "C" KVP_API kvp_status paged_attention_step_noalloc(kvp_pool* pool, const void* q, void* out,
                                                   const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                                   const int32_t* block_tables, int max_blocks_per_seq,
                                                   int num_reqs, int num_tokens, int n_q_heads, int max_q_len,
                                                   int max_context_len, float softmax_scale, kvp_stream stream) {
    if (!pool || num_reqs < 0 || num_tokens < 0) return KVP_E_INVALID_ARG;
    if (num_tokens == 0) return KVP_OK;
    const size_t need = kvp::make_step_layout(num_reqs, num_tokens).total;
    if (need > kNoAllocScratchBytes) return KVP_E_WORKSPACE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVP_E_CUDA;
    // The pool's own device state is made (allocated) by its first kv_append; this entry
    // point never makes it.
    if (kvp::pool_device(pool) != dev) return KVP_E_INVALID_ARG;
    void* scratch = scratch_address(dev);
    if (!scratch) return KVP_E_CUDA;
    return paged_attention_step(pool, q, out, cu_seqlens_q, context_lens, block_tables, max_blocks_per_seq, num_reqs,
                                num_tokens, n_q_heads, max_q_len, max_context_len, softmax_scale, scratch,
                                kNoAllocScratchBytes, stream);
}
