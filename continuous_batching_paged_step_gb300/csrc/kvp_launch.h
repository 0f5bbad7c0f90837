// Host-side interface between the C-ABI layer (kvp_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

struct kvp_pool;

namespace kvp {

// Scratch layout inside the caller's workspace for one paged_attention_step call.
// Offsets are in bytes from the workspace base; every region is 256-byte aligned.
struct StepLayout {
    int max_prefill_tiles;   // (request, 32-token q tile) work items of prefill chunks
    int max_partials;        // split-KV partial slots: request r cut by decode piece p uses r + p
    size_t counters_off;     // int32[8]: 1 = prefill tiles, 2 = decode CTAs, 3 = prefill CTAs done,
                             // 4 = decode chunks taken, 5 = mixed step kernel tickets taken,
                             // 6 = prefill work items claimed
    size_t page_off_off;     // int32 [num_reqs + 1]: first global decode block of each request
    size_t prefill_tiles_off;// int4 {r, first token of tile, tokens in tile, 0}
    size_t part_acc_off;     // float [slot][32 heads][128]  (unnormalised)
    size_t part_ml_off;      // float2 [slot][32 heads]      (running max (log2 units), sum)
    size_t total;
};

// Upper bound of the decode grid (CTAs that share out the decode blocks).
constexpr int kMaxDecodeCtas = 1024;

StepLayout make_step_layout(int num_reqs, int num_tokens);

struct StepArgs {
    const void* q;
    void* out;
    const int32_t* cu_seqlens_q;
    const int32_t* context_lens;
    const int32_t* block_tables;
    int max_blocks_per_seq;
    int num_reqs;
    int num_tokens;
    int max_q_len;
    int max_context_len;
    float softmax_scale;
    const void* k_cache;
    const void* v_cache;
    int num_blocks;
    uint32_t* err;
    char* ws;
    StepLayout lay;
    int num_sms;
    int decode_ctas;   // 0: one CTA per SM
};

cudaError_t launch_kv_append(const void* k_new, const void* v_new, const int32_t* cu, const int32_t* ctx,
                             const int32_t* tables, int max_blocks, int num_reqs, int num_tokens, void* k_cache,
                             void* v_cache, const int32_t* refcnt, int num_blocks, uint32_t* err,
                             cudaStream_t stream);

cudaError_t launch_step_prep(const StepArgs& a, cudaStream_t stream);
cudaError_t launch_decode(const StepArgs& a, const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                          cudaStream_t stream);
// Merge the split-KV partials of decode rows cut into several pieces (after the decode
// kernel and, when there is one, the prefill kernel).
cudaError_t launch_combine(const StepArgs& a, cudaStream_t stream);
cudaError_t launch_prefill(const StepArgs& a, const CUtensorMap* tmap_q, const CUtensorMap* tmap_k,
                           const CUtensorMap* tmap_v, cudaStream_t stream);
// The step's decode rows and prefill tiles in one grid (attn_mixed.cu): the decode
// kernel's CTAs and the prefill kernel's CTAs, each CTA taking the next work ticket.
cudaError_t launch_mixed(const StepArgs& a, const CUtensorMap* tmap_q, const CUtensorMap* tmap_k,
                         const CUtensorMap* tmap_v, const CUtensorMap* tmap_k_blk, const CUtensorMap* tmap_v_blk,
                         cudaStream_t stream);

// Whole-block copies (K and V, 32 KiB each): block i of the launch reads
// src[kv] + (src_ids_used ? src_ids[i] : i) * 32 KiB and writes dst[kv] + (dst_ids_used ?
// dst_ids[i] : i) * 32 KiB, for kv = 0 (K), 1 (V).  Pools are indexed by block id, host
// buffers by position in the list.
constexpr int kMoveChunk = 1024;
struct BlockMoveArgs {
    const uint8_t* src[2];
    uint8_t* dst[2];
    int n;
    int src_ids_used, dst_ids_used;
    int32_t src_ids[kMoveChunk];
    int32_t dst_ids[kMoveChunk];
};
cudaError_t launch_block_move(const BlockMoveArgs& a, cudaStream_t stream);

// Launch `kernel` so that it may start while the previous kernel of `stream` finishes
// (programmatic dependent launch); the kernel must call grid_dep_wait() before it reads
// what earlier kernels wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Device the pool's device-side state lives on, or -1 if it has none yet.
int pool_device(const ::kvp_pool* p);

// One-time per-device kernel attributes (dynamic shared memory limits).
cudaError_t configure_kernels();

// Prefill work unit: a CTA takes 64 query tokens of one request and one KV group, as two
// MMA tiles of 32 tokens x 4 query heads = 128 rows each.
constexpr int kPrefillTileTokens = 64;
constexpr int kPrefillMmaTokens = 32;

}  // namespace kvp
