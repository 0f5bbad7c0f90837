/*
 * kvpaged.h -- C ABI of the GB300 (sm_103a) continuous-batching paged attention step.
 *
 * One packed step of continuous batching: the mixed prefill-chunk and decode rows of
 * this iteration are packed into one flat token matrix (page "Continuous Batching" on
 * k4i.top, section "把 prefill 和 decode 打包在一起"; page "11.2 连续批处理与
 * PagedAttention", section 11.2.2, Figure 11-3).  Their new K/V are appended into a
 * block-paged KV cache, then every packed query row attends to its own request's
 * visible keys only (the block-diagonal causal mask M_ij of the k4i.top page, section
 * "防止跨请求 attention").
 *
 * Fixed geometry of this build: block size 16 tokens, 8 KV heads, 32 query heads (query
 * head h reads KV head h / 4), head_dim 128, bf16 storage, fp32 accumulation.
 *
 * Memory ownership
 *   The caller owns every device buffer passed in (K/V pools, Q, new K/V, metadata,
 *   output, workspace) and every stream.  The library owns the host-side block
 *   allocator, a device mirror of the block refcounts and a device error word; the
 *   device parts are allocated on the first device call of a pool (on the device that
 *   is current then) and freed by kv_pool_destroy.
 *
 * Pool layout (device, caller-allocated, 16-byte aligned):
 *   k_cache, v_cache: bf16 [num_blocks][n_kv_heads = 8][block_size = 16][head_dim = 128]
 *   One (block, head) tile of 16 tokens x 128 dims is 4 KiB contiguous; one block of
 *   all 8 heads is 32 KiB contiguous.  Token slot of logical position p of a request is
 *   block_tables[r][p / 16] * 16 + p % 16 (page "连续批处理与 PagedAttention 原理",
 *   section "block table 与地址映射").
 *
 * Packed step metadata (device int32, caller-allocated):
 *   cu_seqlens_q [num_reqs + 1]: cumulative query rows; request r owns packed rows
 *     cu_seqlens_q[r] .. cu_seqlens_q[r+1]-1 (the cu_seqlens of the varlen attention
 *     interface, page "11.2", section 11.2.2); cu_seqlens_q[0] = 0 and
 *     cu_seqlens_q[num_reqs] = num_tokens.  A request may bring 0 rows.
 *   context_lens [num_reqs]: tokens of request r cached BEFORE this step.  Row j of
 *     request r is at position context_lens[r] + j and sees positions 0 .. that
 *     position of request r (its cached keys, the earlier rows of this step, itself).
 *   block_tables [num_reqs][max_blocks_per_seq]: physical block ids, row-major.
 *
 * Errors
 *   No call aborts, traps or throws.  Host-detectable argument errors return at once
 *   with nothing launched.  Errors found by kernels (bad block id, write into a shared
 *   block, inconsistent metadata, a bounded wait that ran out) set bits in the pool's
 *   device error word; the offending write or tile is skipped and the step's other
 *   outputs are still produced.  kv_pool_get_error() reads and clears the word.
 *
 * Calls are asynchronous on the given stream (NULL = the legacy default stream) unless
 * stated otherwise, and are not thread-safe for one pool.
 */
#ifndef KVPAGED_H
#define KVPAGED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KVP_API __attribute__((visibility("default")))
#else
#define KVP_API
#endif

typedef struct kvp_pool kvp_pool;
/* Same type as cudaStream_t. */
typedef struct CUstream_st* kvp_stream;

typedef enum {
    KVP_OK = 0,
    KVP_E_INVALID_ARG = -1,   /* a host-checked argument is out of range                 */
    KVP_E_NO_BLOCKS = -2,     /* the free list cannot satisfy an allocation               */
    KVP_E_BAD_BLOCK = -3,     /* a block id outside [0, num_blocks) or not allocated      */
    KVP_E_SHARED_WRITE = -4,  /* a write targeted a block whose refcount is not 1         */
    KVP_E_BAD_META = -5,      /* cu_seqlens / context lengths / table width inconsistent  */
    KVP_E_CUDA = -6,          /* a CUDA runtime call failed                               */
    KVP_E_REFCOUNT = -7,      /* free/ref of a block that is not allocated (double free)  */
    KVP_E_WORKSPACE = -8,     /* workspace missing or smaller than required               */
    KVP_E_TIMEOUT = -9        /* a bounded device wait ran out; outputs of that tile lost */
} kvp_status;

/* Bits of the device error word (kv_pool_get_error's *bits). */
#define KVP_ERRBIT_BAD_BLOCK    0x1u
#define KVP_ERRBIT_SHARED_WRITE 0x2u
#define KVP_ERRBIT_BAD_META     0x4u
#define KVP_ERRBIT_TIMEOUT      0x8u

#define KVP_DTYPE_BF16 1

/* ---------------------------------------------------------------- pool lifetime ----
 * kv_pool_create: wrap caller-allocated pools of num_blocks blocks.  block_size must be
 * 16, n_kv_heads 8, head_dim 128, dtype KVP_DTYPE_BF16; k_cache / v_cache are device
 * pointers, 16-byte aligned, each num_blocks * 32 KiB.  All blocks start free.  This
 * call touches no CUDA API (the device state is made on first device use).
 * Physical KV block pool carved once at start-up: page "11.2", section 11.2.3 (steps 1-2);
 * page "连续批处理与 PagedAttention 原理", section "分页设计".
 * Returns KVP_E_INVALID_ARG for bad geometry or NULL pointers. */
KVP_API kvp_status kv_pool_create(int num_blocks, int block_size, int n_kv_heads, int head_dim,
                          int dtype, void* k_cache, void* v_cache, kvp_pool** out);

/* Free the library-owned host and device state (synchronises the device of the pool).
 * The caller's pools are not freed.  NULL is accepted. */
KVP_API kvp_status kv_pool_destroy(kvp_pool* pool);

/* ------------------------------------------------------------ block allocator ------
 * The block manager of page "连续批处理与 PagedAttention 原理" (section "块管理器"): free
 * list plus one refcount per physical block.  All calls are host-only and
 * all-or-nothing: on error nothing changes.  Changes reach the device refcount mirror
 * (used by kv_append's shared-block check) at the next kv_append on any stream, in
 * stream order. */

/* Pop n free blocks (refcount := 1) into out_ids[n] (host memory).  On-demand growth:
 * page "11.2", section 11.2.3 (step 3).  KVP_E_NO_BLOCKS if fewer than n are free. */
KVP_API kvp_status kv_block_alloc(kvp_pool* pool, int n, int32_t* out_ids);

/* Take the n listed blocks out of the free list (refcount := 1).  For placing a step's
 * blocks at chosen physical ids.  KVP_E_BAD_BLOCK if an id is out of range, already
 * allocated or listed twice. */
KVP_API kvp_status kv_block_claim(kvp_pool* pool, int n, const int32_t* ids);

/* Share: refcount += 1 for each listed allocated block (a full prefix block referenced
 * by another request's table, page "11.2", section 11.2.4; page "连续批处理与
 * PagedAttention 原理", section "前缀共享").  KVP_E_REFCOUNT if a block is free. */
KVP_API kvp_status kv_block_ref(kvp_pool* pool, int n, const int32_t* ids);

/* Release: refcount -= 1 per listing; a block returns to the free list at 0 (page "11.2",
 * section 11.2.3, step 4; page "Continuous Batching", section "iteration-level
 * scheduling").  KVP_E_REFCOUNT if a block would go below 0 (double free). */
KVP_API kvp_status kv_block_free(kvp_pool* pool, int n, const int32_t* ids);

/* Copy-on-write (page "11.2", section 11.2.3, the paragraph on sharing: output sequences
 * of one request that share the prompt's last, partly filled block copy it before one of
 * them writes a new token into it; page "连续批处理与 PagedAttention 原理", section
 * "块管理器": copy-on-write is one of the block manager's operations).  For each listed
 * block, in order: if its refcount is 1, out_ids[i] = src_ids[i] and nothing changes;
 * if it is shared, a free block is allocated (refcount := 1), the source's K and V
 * (32 KiB each) are copied into it on `stream`, the source's refcount drops by 1 and
 * out_ids[i] is the new block.  The caller then points its block table at out_ids[i]
 * before writing (kv_append refuses writes into shared blocks).  src_ids / out_ids are
 * host arrays of n.  All-or-nothing on the host: KVP_E_BAD_BLOCK for an id out of range
 * or free, KVP_E_NO_BLOCKS if the free list cannot supply the copies; KVP_E_CUDA if a
 * launch fails (the allocations stand; the copies may be missing).  Launches nothing
 * when no listed block is shared. */
KVP_API kvp_status kv_block_cow(kvp_pool* pool, int n, const int32_t* src_ids, int32_t* out_ids,
                                kvp_stream stream);

/* Swap out (page "Continuous Batching 深入实现", section "第四层：Preemption 与 Recompute
 * vs Swap": a preempted request's KV is copied from HBM to host memory and its GPU
 * blocks are released; page "连续批处理与 PagedAttention 原理", section "抢占策略").
 * Block ids[i]'s K and V go to host_k + i * 32 KiB and host_v + i * 32 KiB, then one
 * reference of each listed block is released (as kv_block_free).  host_k / host_v: page-
 * locked host memory (cudaHostAlloc / cudaHostRegister) of at least n * 32 KiB, written
 * by a kernel on `stream`; they hold the data once the stream has passed this call.  The
 * released blocks may be handed out again at once: later writes to them must be ordered
 * after this call (same stream, or after synchronising it).  KVP_E_BAD_BLOCK /
 * KVP_E_REFCOUNT as kv_block_free, KVP_E_INVALID_ARG if a host buffer is not page-locked
 * memory the device can reach (nothing changes then). */
KVP_API kvp_status kv_blocks_swap_out(kvp_pool* pool, int n, const int32_t* ids, void* host_k,
                                      void* host_v, kvp_stream stream);

/* Swap in (same passages: the KV is copied back when the request resumes): allocate n
 * blocks (refcount := 1) into out_ids[n] (host) and copy host_k + i * 32 KiB /
 * host_v + i * 32 KiB into block out_ids[i] on `stream` (page-locked host memory as for
 * kv_blocks_swap_out, which must stay unchanged until the stream has passed this call).
 * The caller writes out_ids into the request's block table.  KVP_E_NO_BLOCKS if fewer
 * than n blocks are free, KVP_E_INVALID_ARG for host buffers the device cannot reach
 * (nothing changes then). */
KVP_API kvp_status kv_blocks_swap_in(kvp_pool* pool, int n, const void* host_k, const void* host_v,
                                     int32_t* out_ids, kvp_stream stream);

/* Number of free blocks, or -1 for NULL. */
KVP_API int kv_pool_num_free(const kvp_pool* pool);

/* Refcount of one block (0 = free), or -1 for a bad id / NULL pool. */
KVP_API int kv_block_refcount(const kvp_pool* pool, int32_t id);

/* ------------------------------------------------------------------- kv_append -----
 * Write this step's new K/V rows into the pool (page "Continuous Batching", section
 * "一个完整的 mixed iteration", the step that stores the current K/V in the owning
 * request's cache;
 * page "11.2", section 11.2.2: the new K and V are appended to the owning request's
 * cache).  For packed row i of request r, position p = context_lens[r] + (i -
 * cu_seqlens_q[r]); for every KV head h the 256-byte row k_new[i][h*128 : h*128+128]
 * goes to k_cache[b][h][p % 16][:] with b = block_tables[r][p / 16]; same for V.
 *   k_new, v_new: device bf16 [num_tokens][8 * 128], row-major.
 * The write is a bit copy.  Device-checked: b in [0, num_blocks) and allocated
 * (KVP_ERRBIT_BAD_BLOCK), refcount(b) == 1 (KVP_ERRBIT_SHARED_WRITE: shared prefix blocks
 * are read-only; copy-on-write belongs to the caller), p / 16 < max_blocks_per_seq and
 * the row lies inside cu_seqlens_q (KVP_ERRBIT_BAD_META); an offending row-head write is
 * skipped.  num_tokens == 0 launches nothing. */
KVP_API kvp_status kv_append(kvp_pool* pool, const void* k_new, const void* v_new,
                     const int32_t* cu_seqlens_q, const int32_t* context_lens,
                     const int32_t* block_tables, int max_blocks_per_seq,
                     int num_reqs, int num_tokens, kvp_stream stream);

/* --------------------------------------------------------- paged attention step ----
 * Workspace bytes paged_attention_step needs for a step with at most these sizes (the
 * same for every pool and decode split); 0 for bad arguments. */
KVP_API size_t paged_attention_workspace_size(const kvp_pool* pool, int num_reqs, int num_tokens,
                                      int n_q_heads, int max_context_len);

/* Varlen paged attention over one packed step (page "Continuous Batching", sections
 * "防止跨请求 attention", "与 KV cache 的关系" (decode formula) and "为什么 packed forward
 * 等价" (visible set S(i)); page "Continuous Batching 深入实现", section "第二层" (cu_seqlens)
 * and "第三层" (a chunk attends to earlier chunks through the cache)).
 *   q:   device bf16 [num_tokens][32 * 128]; out: device bf16 [num_tokens][32 * 128].
 *   For row i of request r at position P and query head h:
 *     out[i][h] = sum_{t<=P} softmax_t(q[i][h] . K_r[t][h/4] * softmax_scale) V_r[t][h/4]
 *   where K_r[t] is read from the pool through block_tables[r] (so kv_append of this
 *   step must precede this call in stream order).  fp32 accumulation; out rounded once
 *   to bf16 (nearest even).
 *   n_q_heads must be 32.  max_q_len / max_context_len must bound the step's values
 *   (KVP_ERRBIT_BAD_META and the request is skipped otherwise).  softmax_scale is
 *   usually 1/sqrt(128).  workspace: device, 256-byte aligned, at least
 *   paged_attention_workspace_size(num_reqs, num_tokens, 32, max_context_len) bytes,
 *   scratch owned by the caller for the duration of the call (stream order).
 * Rows with q_len == 1 (decode) take the HBM-bound split-KV path; rows of requests with
 * q_len > 1 (prefill chunks) take the tcgen05 tensor-core path.  The two kernels run side
 * by side on disjoint SMs (the step's first kernel sizes the decode's share from the
 * step's work); a last kernel merges the partial results of decode rows that the split
 * cut into pieces.  The call's work is complete, in stream order, when that kernel is. */
KVP_API kvp_status paged_attention_step(kvp_pool* pool, const void* q, void* out,
                                const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                const int32_t* block_tables, int max_blocks_per_seq,
                                int num_reqs, int num_tokens, int n_q_heads, int max_q_len,
                                int max_context_len, float softmax_scale, void* workspace,
                                size_t workspace_bytes, kvp_stream stream);

/* Decode split: the 16-token blocks of all decode rows of a step are shared out evenly,
 * in request order, among `ctas` CTAs at a time (0 = one per SM, the default; at most
 * 1024; a step that also has prefill chunks gives the decode at most the share of SMs its
 * metadata kernel leaves it); a CTA's range holds at most 1,024 blocks, so a step with
 * more than ctas x 1,024 decode blocks runs in several waves of CTAs (at most 1024 CTAs in
 * all: a step whose decode rows hold more blocks than that allows sets
 * KVP_ERRBIT_BAD_META).  The last fifth of each range is handed out in small chunks to
 * whichever CTA runs out of work first, so that SMs that stream more slowly finish with
 * the others.  A row whose blocks fall to several pieces (ranges or chunks) is finished by
 * a merge of their partial results.  The workspace size does not depend on this setting.
 * Host-only. */
KVP_API kvp_status kv_pool_set_decode_ctas(kvp_pool* pool, int ctas);

/* Synchronise `stream`, then read and clear the pool's device error word.  *bits (may be
 * NULL) receives the KVP_ERRBIT_* mask; the return value is KVP_OK for an empty word,
 * else the status of the lowest set bit (BAD_BLOCK, SHARED_WRITE, BAD_META, TIMEOUT). */
KVP_API kvp_status kv_pool_get_error(kvp_pool* pool, kvp_stream stream, uint32_t* bits);

/* ---------------------------------------------------------- allocation-free step ----
 * The pages have no counterpart: this is a convenience of this library.
 * Same as paged_attention_step, but without a caller workspace: for callers that cannot
 * allocate device memory at step time (an engine that gave all free device memory to
 * its KV pool, or a serving loop that must not call cudaMalloc/cudaFree because they can
 * synchronise the device).  The scratch lives in a fixed device array inside the library
 * (paged_attention_noalloc_capacity() bytes, 32 MiB), held by every GPU that loads the
 * library until the process exits.  It holds the scratch of a step of at most about 990
 * requests (991 for a decode-only step): every request and each of the decode kernel's up
 * to 1,024 pieces has a slot of split-KV partials of about 16.6 KiB.  The call allocates nothing: the pool must already
 * have its device state (made by its first kv_append on the current device), else
 * KVP_E_INVALID_ARG.  A step whose scratch (paged_attention_workspace_size) exceeds the
 * array is rejected with KVP_E_WORKSPACE before anything is launched.  All calls share
 * the array: calls whose kernels overlap on the GPU (other streams, other threads) race
 * on it; calls on one stream are ordered.  Nothing in it needs to start at zero.  The
 * first call with a given device current looks the array's device address up
 * (cudaGetSymbolAddress); make it before any stream capture begins. */
KVP_API kvp_status paged_attention_step_noalloc(kvp_pool* pool, const void* q, void* out,
                                                const int32_t* cu_seqlens_q,
                                                const int32_t* context_lens,
                                                const int32_t* block_tables, int max_blocks_per_seq,
                                                int num_reqs, int num_tokens, int n_q_heads,
                                                int max_q_len, int max_context_len,
                                                float softmax_scale, kvp_stream stream);

/* Bytes of the fixed scratch array used by paged_attention_step_noalloc. */
KVP_API size_t paged_attention_noalloc_capacity(void);

/* ------------------------------------------------------------------ diagnostics ----
 * Per-kernel timing of the library's own launches, for benchmarks.  After
 * kv_pool_enable_timing(pool, max_launches) every kernel launch of kv_append,
 * paged_attention_step and the block copies (on this pool's device) is bracketed by two
 * CUDA events on the launching stream, up to max_launches launches (0 disables and frees
 * the events).
 * kv_pool_read_timing waits for the last recorded event, writes the number of timed
 * launches and the summed milliseconds of each kernel kind into counts[KVP_NUM_KERNELS]
 * and ms[KVP_NUM_KERNELS], and restarts the record. */
#define KVP_KERNEL_APPEND  0
#define KVP_KERNEL_PREP    1
#define KVP_KERNEL_PREFILL 2
#define KVP_KERNEL_DECODE  3   /* split-KV partials of decode rows cut into several pieces */
#define KVP_KERNEL_BLOCKS  4   /* block copies of kv_block_cow / kv_blocks_swap_* */
#define KVP_KERNEL_COMBINE 5   /* merges those partials */
#define KVP_KERNEL_MIXED   6   /* the mixed step kernel (decode rows and prefill tiles in one grid) */
#define KVP_NUM_KERNELS    7
KVP_API kvp_status kv_pool_enable_timing(kvp_pool* pool, int max_launches);
KVP_API kvp_status kv_pool_read_timing(kvp_pool* pool, int* counts, float* ms);

/* Which kernels run a step's attention: 0 (the default) launches the decode kernel and the
 * prefill kernel as its programmatic dependent, side by side on disjoint SMs; 1 launches
 * the mixed step kernel, one persistent grid whose CTAs take a work ticket from a device
 * counter in the order they start (the decode CTAs' block ranges go to the first tickets)
 * and then take prefill (tile, KV head) items, longest first, from another counter until
 * none are left (page "Continuous Batching", section "把 prefill 和 decode 打包在一起": one
 * packed pass).  The results are the same up to the order of floating-point
 * additions (identical per row: both run the same CTA code).  KVP_E_INVALID_ARG for
 * another value or a null pool.  Host-side setting, no device work. */
KVP_API kvp_status kv_pool_set_step_kernel(kvp_pool* pool, int mixed);

/* NVTX ranges (domain "kvpaged"): with on != 0, kv_append, paged_attention_step, the
 * block copies and every kernel launch of this pool are wrapped in named ranges
 * (kv_append, paged_attention_step, kv_append_kernel, step_prep_kernel, decode_kernel,
 * prefill_kernel, combine_kernel, block_move_kernel) so a profiler's timeline shows them;
 * off by default.  Without a profiler attached the ranges cost next to nothing.
 * KVP_E_INVALID_ARG for a null pool. */
KVP_API kvp_status kv_pool_set_nvtx(kvp_pool* pool, int on);

/* Number of kernels this pool's calls have launched so far (host counter). */
KVP_API long long kv_pool_launch_count(const kvp_pool* pool);

/* Make one bounded device wait run out on purpose: a single thread waits on an mbarrier
 * that nothing arrives at, for limit_ns nanoseconds (0 < limit_ns <= 2e9), on `stream`
 * (synchronised before returning).  Returns KVP_E_TIMEOUT when the wait gave up as it
 * should (the same bounded-wait mechanism the step's kernels use, which then set
 * KVP_ERRBIT_TIMEOUT and finish), KVP_OK if the barrier completed (it cannot), or
 * KVP_E_INVALID_ARG / KVP_E_CUDA.  Faults and hangs nothing; allocates 4 bytes. */
KVP_API kvp_status kvp_selftest_bounded_wait(long long limit_ns, kvp_stream stream);

/* Human-readable name of a status code (static storage). */
KVP_API const char* kvp_status_string(kvp_status s);

#ifdef __cplusplus
}
#endif

#endif /* KVPAGED_H */
