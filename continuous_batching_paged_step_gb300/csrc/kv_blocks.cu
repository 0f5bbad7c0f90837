// Whole-block copies for the block manager: copy-on-write of a shared block (page "11.2
// 连续批处理与 PagedAttention", section 11.2.3, sharing within one request; page "连续批
// 处理与 PagedAttention 原理", section "块管理器") and swapping a preempted request's
// blocks out to host memory and back (page "Continuous Batching 深入实现", section "第四
// 层：Preemption 与 Recompute vs Swap").
//
// One block of all 8 KV heads is 32 KiB contiguous in the K pool and again in the V pool,
// so a block moves as two contiguous 32 KiB copies.  One CTA of 256 threads per (block,
// K|V): each thread moves 8 chunks of 16 bytes, consecutive threads on consecutive chunks
// (fully coalesced on both sides).  Host buffers are page-locked memory the kernel reads or
// writes directly (over the CPU-GPU link), so a swap needs no device staging buffer.  The
// block ids travel in the kernel's parameters (up to kMoveChunk per launch), so nothing
// is allocated or uploaded for them.
#include "kvp_device.cuh"
#include "kvp_launch.h"

namespace kvp {

namespace {

__global__ void __launch_bounds__(256) block_move_kernel(const BlockMoveArgs a) {
    const int i = blockIdx.x, kv = blockIdx.y;
    const size_t src_blk = a.src_ids_used ? (size_t)a.src_ids[i] : (size_t)i;
    const size_t dst_blk = a.dst_ids_used ? (size_t)a.dst_ids[i] : (size_t)i;
    const uint4* src = reinterpret_cast<const uint4*>(a.src[kv] + src_blk * kBlockBytes);
    uint4* dst = reinterpret_cast<uint4*>(a.dst[kv] + dst_blk * kBlockBytes);
    constexpr int kChunks = kBlockBytes / 16;
    uint4 v[kChunks / 256];
#pragma unroll
    for (int j = 0; j < kChunks / 256; ++j) v[j] = src[j * 256 + threadIdx.x];
#pragma unroll
    for (int j = 0; j < kChunks / 256; ++j) dst[j * 256 + threadIdx.x] = v[j];
}

}  // namespace

cudaError_t launch_block_move(const BlockMoveArgs& a, cudaStream_t stream) {
    if (a.n <= 0) return cudaSuccess;
    block_move_kernel<<<dim3(a.n, 2), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace kvp
