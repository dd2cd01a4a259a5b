/*
 * pa.h -- C ABI of libpa: PagedAttention decode on one GB300 (sm_103a).
 *
 * The library implements the one data-parallel hot path the pages on vLLM
 * turn on: for each running sequence, one fp16 query per head attends over
 * that sequence's K/V history, o = softmax(scale * K q)^T V
 * ("vLLM 2026 推理引擎全解：从 PagedAttention 到分离式 Prefill", §1.1).  The
 * history lives in fixed-size KV blocks scattered through device memory and is
 * reached through a per-sequence block table (logical block -> physical
 * block); blocks may be shared between sequences with a common prompt prefix
 * (same page, §2.1 and §2.3; mjmagnets.cn vLLM tutorial, §2.1-§2.2).
 *
 * Conventions for every call:
 *  - Pointers marked "device" must point to device memory of the current CUDA
 *    device (or memory the device can read, such as managed memory); pointers
 *    marked "host" are read on the host during the call only.
 *  - The caller owns every buffer.  The library keeps no pointer past the call.
 *  - All work is enqueued on `stream` (a cudaStream_t; NULL means the legacy
 *    default stream) and runs asynchronously: a PA_OK return means the launch
 *    succeeded, not that the kernel has finished.
 *  - 16-bit tensors (fp16 or bf16, per pa_dims.dtype) are row-major and
 *    contiguous in the shapes given; every such device pointer must be
 *    16-byte aligned.
 *  - Errors found on the host return a negative pa_status and launch nothing.
 *    Errors only the device can see (a block-table entry or slot outside the
 *    pool, a context length outside [0, max_blocks_per_seq * block_size]) are
 *    recorded in a per-device error word, read with pa_device_errors(); the
 *    kernels skip the offending access instead of faulting.
 *  - No call aborts, throws or traps.
 *  - The library caches per-device state on first use (device addresses of
 *    its error word and scratch array, kernel attributes).  A
 *    cudaDeviceReset, or anything else that destroys the device's primary
 *    context, invalidates that state: the library must not be called on that
 *    device afterwards within the same process.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_NULL = -1,          /* a required pointer is NULL                    */
    PA_ERR_SHAPE = -2,         /* a size is negative, zero where it must not be, or overflows */
    PA_ERR_UNSUPPORTED = -3,   /* head_dim / block_size / dtype outside the built variants,
                                  or memory the device cannot address */
    PA_ERR_ALIGN = -4,         /* an fp16 pointer is not 16-byte aligned        */
    PA_ERR_WORKSPACE = -5,     /* workspace or counter buffer missing, too small or misaligned */
    PA_ERR_CUDA = -6,          /* a CUDA runtime call failed; see pa_last_cuda_error() */
    PA_ERR_OUT_OF_BLOCKS = -7  /* the KV block manager's free list is empty             */
} pa_status;

/* Bits of the per-device error word (pa_device_errors). */
#define PA_DEVERR_TABLE   0x1u  /* a used block-table entry was outside [0, num_blocks)   */
#define PA_DEVERR_CONTEXT 0x2u  /* a context length was < 0 or > max_blocks_per_seq * block_size */
#define PA_DEVERR_SLOT    0x4u  /* a slot_mapping entry was >= num_blocks * block_size      */
#define PA_DEVERR_TIMEOUT 0x8u  /* an internal pipeline wait gave up (should never happen) */
#define PA_DEVERR_PREFIX  0x10u /* pa_decode_shared_prefix: a sequence could not use its group's
                                   shared prefix (see there) and was decoded in full instead */

/* Element type of q, the caches and the output (and of k, v for
 * reshape_and_cache): IEEE binary16, or bfloat16 (the top 16 bits of an
 * IEEE binary32).  The pages name both for the kernels (doramagic.ai vLLM
 * manual, "PagedAttention V1 内核": FP16/BF16). */
typedef enum pa_dtype {
    PA_DTYPE_F16 = 0,
    PA_DTYPE_BF16 = 1
} pa_dtype;

/* Sizes shared by both calls.
 *   num_seqs    S: sequences in the decode batch (>= 0)
 *   num_heads   H: attention heads; K/V heads equal query heads (no grouping)
 *   head_dim    D: 64, 128 or 256
 *   block_size  B: tokens per KV block: 8, 16 (the pages' default) or 32
 *   num_blocks  N: physical blocks in the cache pool (> 0)
 *   dtype       a pa_dtype; a zero-initialised struct selects fp16
 * Cache layout [N, H, B, D] fp16: element (blk, h, t, d) is at
 * ((blk * H + h) * B + t) * D + d ("vLLM 2026 推理引擎全解", §2.2, the kernel
 * sketch's k_cache layout [num_pages, num_heads, page_size, head_dim]). */
typedef struct pa_dims {
    int32_t num_seqs;
    int32_t num_heads;
    int32_t head_dim;
    int32_t block_size;
    int32_t num_blocks;
    int32_t dtype;
} pa_dims;

/*
 * pa_reshape_and_cache -- store each new token's K and V in its cache slot.
 *
 * Source: the step that caches K and V for reuse and appends each new token
 * to the KV cache ("vLLM 2026 推理引擎全解", §1.1; doramagic.ai vLLM manual,
 * "KVCacheManager 缓存管理": 追加新Token).  The slot encoding is not given by
 * the pages; this library reads slot = physical_block * B + offset.
 *
 *   k, v          device, fp16 [num_tokens, H, D]: the new tokens' keys / values
 *   k_cache       device, fp16 [N, H, B, D]: updated in place
 *   v_cache       device, fp16 [N, H, B, D]: updated in place
 *   slot_mapping  device, int32 [num_tokens]: slot of token i; slot < 0 skips
 *                 the token; slot >= N * B is skipped and flags PA_DEVERR_SLOT
 *   num_tokens    >= 0 (0 launches nothing)
 *   dims          host; num_seqs is not used
 *   stream        cudaStream_t
 *
 * For each i with 0 <= slot < N*B and every head h:
 *   k_cache[slot / B, h, slot % B, :] = k[i, h, :]   (same for v)
 * Copies are bit-exact.  Two tokens mapping to the same slot race.
 */
int pa_reshape_and_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                         const int32_t *slot_mapping, int32_t num_tokens,
                         const pa_dims *dims, void *stream);

/*
 * pa_copy_blocks -- copy whole KV blocks between two block pools.
 *
 * Source: the KV cache manager's block moves -- blocks shared between
 * requests through reference counts, so a request that must change a shared
 * block gets its own copy, and blocks swapped out to CPU memory when GPU
 * memory runs short and swapped back in later (doramagic.ai vLLM manual,
 * "内存管理策略", "BlockPool 组件", "共享机制").  One call covers copy-on-write
 * (source pool = destination pool), swap-out (device -> host) and swap-in
 * (host -> device).
 *
 *   src_k, src_v    [src_num_blocks, H, B, D] 16-bit elements: the source pool
 *   dst_k, dst_v    [dst_num_blocks, H, B, D]: the destination pool (written)
 *   block_pairs     device (or device-addressable), int32 [num_pairs][2]:
 *                   (source block, destination block)
 *   num_pairs       >= 0 (0 launches nothing)
 *   dims            host; num_heads, head_dim, block_size and dtype are used
 *   stream          cudaStream_t
 *
 * Every pool pointer must be memory the current device can address in a
 * kernel: its own device memory, managed memory, pinned or registered host
 * memory (cudaHostAlloc / cudaHostRegister), or any host memory when the
 * device reports cudaDevAttrPageableMemoryAccess.  Anything else returns
 * PA_ERR_UNSUPPORTED before launching.  For each pair, K and V of block src
 * (all heads) are copied bit for bit to block dst.  A pair with an id outside
 * its pool is skipped and sets PA_DEVERR_TABLE.  Destinations must be
 * distinct and must not be the source of another pair (such copies race).
 */
int pa_copy_blocks(const void *src_k, const void *src_v, int32_t src_num_blocks, void *dst_k,
                   void *dst_v, int32_t dst_num_blocks, const int32_t *block_pairs,
                   int32_t num_pairs, const pa_dims *dims, void *stream);

/*
 * pa_decode -- paged-attention decode for a batch of sequences.
 *
 * Source: o = Attention(q_t, K_{1:t}, V_{1:t}) ("vLLM 2026 推理引擎全解",
 * §1.1), with K/V gathered block by block through the block table
 * (mjmagnets.cn vLLM tutorial, §2.2; "vLLM 2026 推理引擎全解", §2.2, where the
 * attention is computed page by page as a paged extension of FlashAttention).
 *
 *   out           device, fp16 [S, H, D]: written.  It may also be pinned or
 *                 registered host memory (the output rows then go straight to
 *                 the host over the host link, written by the kernel as each
 *                 row completes); the caller reads it after the stream has
 *                 reached the end of the call
 *   q             device, fp16 [S, H, D]: one query per sequence and head
 *   k_cache       device, fp16 [N, H, B, D]
 *   v_cache       device, fp16 [N, H, B, D]
 *   block_tables  device, int32 [S, max_blocks_per_seq]: logical -> physical
 *                 block; only the first ceil(ctx_s / B) entries of row s are
 *                 read, so the rest may hold anything
 *   context_lens  device, int32 [S]: ctx_s, tokens of sequence s (0 gives a
 *                 zero output row)
 *   scale         softmax scale (1/sqrt(D) for standard attention)
 *   max_blocks_per_seq  row length of block_tables (> 0)
 *   dims, stream  as above
 *
 * For each s, h:  out[s,h,:] = sum_t softmax_t(scale * q[s,h,:] . K_t) V_t
 * over t < ctx_s, where K_t / V_t is row t % B of block
 * block_tables[s, t / B] at head h.  Scores, the running max/sum softmax and
 * the weighted sum are fp32; the output is rounded to fp16 (nearest even).
 *
 * Long contexts are split into partitions processed in parallel and combined
 * on the device (by the last partition of each (sequence, head) to finish, in
 * the same launch).  This call allocates its counter buffer and partial-result
 * workspace itself with stream-ordered cudaMallocAsync / cudaFreeAsync (and
 * zeroes the counters with cudaMemsetAsync); pa_decode_ws takes them from the
 * caller instead.
 */
int pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_tables, const int32_t *context_lens, float scale,
              int32_t max_blocks_per_seq, const pa_dims *dims, void *stream);

/*
 * pa_prefill -- causal multi-query attention over the paged cache (prefill).
 *
 * Source: prefill processes a prompt's tokens together and is compute-bound
 * ("vLLM 2026 推理引擎全解", §1.3); each token attends to itself and the
 * tokens before it, o_t = Attention(q_t, K_{1:t}, V_{1:t}) (same page, §1.1),
 * with K/V gathered through the block table (§2.1-§2.2).  Runs on the tcgen05
 * tensor cores (S = Q K^T and P V in tensor memory).
 *
 *   out           device, [total_query_tokens, H, D] (written)
 *   q             device, [total_query_tokens, H, D]
 *   k_cache, v_cache, block_tables, context_lens: as pa_decode; the queries'
 *                 own K/V must already be in the cache (pa_reshape_and_cache)
 *   query_start   device, int32 [S + 1]: sequence s owns query rows
 *                 query_start[s] .. query_start[s + 1] - 1, which are the last
 *                 q_len_s = query_start[s + 1] - query_start[s] tokens of its
 *                 context (a whole prompt, or its latest chunk)
 *   total_query_tokens  host: rows of q and out
 *   max_query_len host: an upper bound of every q_len_s (sizes the work)
 *   scale, max_blocks_per_seq, dims, stream: as pa_decode
 *
 * Query i of sequence s sits at position p = ctx_s - q_len_s + i and
 * attends to keys 0 .. p.  Built for head_dim 128, block_size 16, fp16 or
 * bf16 (PA_ERR_UNSUPPORTED otherwise).  Scores and softmax are fp32; the
 * probabilities enter the P V product as a pair of 16-bit values (P_hi +
 * P_lo, P_hi the weight rounded to 16 bits and P_lo the rounded remainder) so
 * the product keeps about 22 bits.  A sequence with q_len_s >
 * ctx_s, ctx_s > max_blocks_per_seq * B, or rows outside
 * [0, total_query_tokens) is skipped and flags PA_DEVERR_CONTEXT; so does a
 * q_len_s above max_query_len rounded up to 256 (its rows past that are not
 * computed).
 *
 * The kernel is persistent (one CTA per SM) and takes its work items from a
 * queue in two device counters; pa_prefill allocates them stream-ordered
 * (cudaMallocAsync) for each call.  PA_ERR_SHAPE if ceil(max_query_len / 256)
 * * S * H exceeds INT32_MAX.
 */
int pa_prefill(void *out, const void *q, const void *k_cache, const void *v_cache,
               const int32_t *block_tables, const int32_t *context_lens,
               const int32_t *query_start, int32_t total_query_tokens, int32_t max_query_len,
               float scale, int32_t max_blocks_per_seq, const pa_dims *dims, void *stream);

/* Bytes of the counters pa_prefill_ws takes. */
#define PA_PREFILL_COUNTERS_BYTES 8

/*
 * pa_prefill_ws -- pa_prefill with caller-owned work-queue counters and no
 * allocation.  counters: device, PA_PREFILL_COUNTERS_BYTES bytes (at least),
 * 4-byte aligned, all zero on entry; the kernel leaves them zero on exit, so
 * one buffer serves every call on one stream.  Two launches that run at the
 * same time (different streams) must not share it.  PA_ERR_WORKSPACE if
 * counters_bytes is too small.
 */
int pa_prefill_ws(void *out, const void *q, const void *k_cache, const void *v_cache,
                  const int32_t *block_tables, const int32_t *context_lens,
                  const int32_t *query_start, int32_t total_query_tokens, int32_t max_query_len,
                  float scale, int32_t max_blocks_per_seq, const pa_dims *dims,
                  uint32_t *counters, size_t counters_bytes, void *stream);

/*
 * Bytes of partial-result workspace pa_decode_ws needs for these sizes and
 * partition length (partition_tokens = 0 selects the default).  0 means no
 * partials are needed (every sequence fits one partition).  Returns
 * (size_t)-1 on invalid sizes.
 */
size_t pa_decode_workspace_bytes(const pa_dims *dims, int32_t max_blocks_per_seq,
                                 int32_t partition_tokens);

/*
 * Bytes of the counter buffer pa_decode_ws needs: a work-queue head, a
 * finished-CTA count and one ticket per (sequence, head), rounded up to 256.
 * Returns 0 on invalid sizes.
 */
size_t pa_decode_counters_bytes(const pa_dims *dims);

/*
 * pa_decode_ws -- pa_decode with caller-provided buffers.
 *
 *   partition_tokens  tokens per context partition: a positive multiple of
 *                     block_size, or 0 for the default.  A value of at least
 *                     max_blocks_per_seq * B processes every sequence in one
 *                     pass with no partial results.
 *   workspace         device, at least pa_decode_workspace_bytes(...) bytes,
 *                     16-byte aligned; holds the partitions' partial results.
 *                     Needs no initialisation.  May be NULL when the required
 *                     size is 0.
 *   workspace_bytes   its size
 *   counters          device, at least pa_decode_counters_bytes(dims) bytes,
 *                     4-byte aligned, ALL ZERO before the first call.  Every
 *                     call that completes without a device error leaves it
 *                     all zero again, so one zeroed counter buffer serves any
 *                     number of calls of any sizes (up to its capacity).
 *                     Calls sharing a counter buffer or a workspace must not
 *                     overlap on the device (use one pair per stream).  After
 *                     a device error (pa_device_errors() != 0), zero the
 *                     counter buffer before reusing it.
 *   counters_bytes    its size
 */
int pa_decode_ws(void *out, const void *q, const void *k_cache, const void *v_cache,
                 const int32_t *block_tables, const int32_t *context_lens, float scale,
                 int32_t max_blocks_per_seq, const pa_dims *dims, int32_t partition_tokens,
                 void *workspace, size_t workspace_bytes, uint32_t *counters,
                 size_t counters_bytes, void *stream);

/*
 * pa_decode_shared_prefix_ws -- pa_decode for a batch in which groups of
 * sequences share the first blocks of their block tables: a common system
 * prompt, or several samples forked from one prompt ("vLLM 2026
 * 推理引擎全解", §2.3: the shared prefix is stored once and referenced by every
 * request; doramagic.ai vLLM manual, "共享机制").  The output is that of
 * pa_decode (within the decode tolerance); what changes is the work.  The
 * pages share the prefix's memory; this call also shares its reads: the
 * prefix's K/V are read once per group and head instead of once per sequence.
 *
 *   out, q, k_cache, v_cache, block_tables, context_lens, scale,
 *   max_blocks_per_seq, dims, partition_tokens: as pa_decode_ws
 *   group_start          device, int32 [num_groups + 1], non-decreasing
 *                        within [0, S]: group g is the sequences
 *                        group_start[g] .. group_start[g + 1] - 1 (sequences
 *                        outside every group are decoded as by pa_decode)
 *   group_prefix_blocks  device, int32 [num_groups]: P_g, the number of
 *                        leading block-table entries every sequence of group g
 *                        shares with the group's first sequence (0: none)
 *   num_groups           host, >= 0
 *   max_group_size       host: an upper bound of the group sizes (sizes the
 *                        prefix work)
 *   workspace            device, pa_decode_shared_prefix_workspace_bytes(...)
 *                        bytes (never 0), 16-byte aligned, no initialisation
 *   counters             device, pa_decode_shared_prefix_counters_bytes(dims)
 *                        bytes, 4-byte aligned, all zero before the first call
 *                        and left zero by every call that completes without a
 *                        device error (as pa_decode_ws)
 *
 * Two launches on `stream` (when num_groups or max_group_size is 0, only
 * pa_decode's):
 *  1. The tcgen05 prefill kernel, in a non-causal mode: for each group, head
 *     and tile of up to 128 member queries, S = Q K^T and P V over the
 *     group's P_g * B prefix keys (read through the group's first sequence's
 *     table), written as one partial result -- (max, sum) and the
 *     unnormalised output -- per member and head.
 *  2. The decode kernel: each member's blocks P_g .. ceil(ctx_s / B) - 1,
 *     merged with the prefix partial by the split-context combine.  It
 *     starts while the prefill kernel still runs (programmatic dependent
 *     launch; that kernel waited for the inputs before letting it start) and
 *     waits for it only before the merges that read a prefix partial, which
 *     each warp makes after its last work unit.
 *
 * A member is decoded in full, as by pa_decode, and PA_DEVERR_PREFIX is set,
 * when its first P_g table entries differ from the group's first sequence's,
 * its context is shorter than P_g * B, it lies past max_group_size rounded up
 * to 256 within its group, or the group arrays are malformed (decreasing,
 * outside [0, S], or P_g outside [0, max_blocks_per_seq]).  Outputs are
 * therefore always those of pa_decode; the flag reports the wasted work.
 *
 * Built for head_dim 128 and block_size 16, fp16 or bf16 (the prefill
 * kernel's shapes); PA_ERR_UNSUPPORTED otherwise.  The prefix keys enter
 * P V as a 16-bit pair (about 22 bits), as in pa_prefill.
 */
size_t pa_decode_shared_prefix_workspace_bytes(const pa_dims *dims, int32_t max_blocks_per_seq,
                                               int32_t partition_tokens);
size_t pa_decode_shared_prefix_counters_bytes(const pa_dims *dims);
int pa_decode_shared_prefix_ws(void *out, const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *block_tables, const int32_t *context_lens,
                               float scale, int32_t max_blocks_per_seq, const pa_dims *dims,
                               const int32_t *group_start, const int32_t *group_prefix_blocks,
                               int32_t num_groups, int32_t max_group_size,
                               int32_t partition_tokens, void *workspace, size_t workspace_bytes,
                               uint32_t *counters, size_t counters_bytes, void *stream);

/*
 * pa_decode_shared_prefix -- pa_decode_shared_prefix_ws with its counters and
 * workspace allocated stream-ordered (cudaMallocAsync / cudaFreeAsync, the
 * counters zeroed with cudaMemsetAsync) for the call, and the default
 * partition length.
 */
int pa_decode_shared_prefix(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, const int32_t *context_lens, float scale,
                            int32_t max_blocks_per_seq, const pa_dims *dims,
                            const int32_t *group_start, const int32_t *group_prefix_blocks,
                            int32_t num_groups, int32_t max_group_size, void *stream);

/* Capacity of the scratch array pa_decode_static uses instead of allocating. */
#define PA_STATIC_SCRATCH_BYTES ((size_t)16 << 20) /* 16 MiB per device */

/*
 * pa_decode_static -- pa_decode that allocates no device memory.
 *
 * The pages have no counterpart: this entry point exists for callers that
 * cannot let a library call cudaMalloc -- a serving process that reserves
 * nearly all device memory for its KV-block pool up front and forbids later
 * allocations, a latency-critical decode loop that must not stall on
 * cudaMalloc / cudaFree (both may synchronise the device), or a plugin in a
 * host program whose allocator it does not control.  The caller passes the
 * same inputs and output as pa_decode; the split-context counters and partial
 * results live in a fixed per-device array of PA_STATIC_SCRATCH_BYTES inside
 * the library, which every GPU that loads the library holds until exit.
 *
 *   Arguments, layouts and results: as pa_decode.  Outputs match pa_decode
 *   within the decode tolerance (the partition length may differ, see below).
 *   Set-up: the first call on a device, made with that device current, looks
 *   up the array's device address (cudaGetSymbolAddress); make that first
 *   call before any stream capture.
 *   Every call zeroes the array's counter area with cudaMemsetAsync on
 *   `stream` and then launches the decode kernel; no cudaMalloc, cudaFree or
 *   other allocating call is made.
 *   Partition length: the pa_decode default when its partial results fit in
 *   the array, otherwise the smallest power-of-two multiple of 512 tokens
 *   that fits, or one pass over each whole context (no partials).
 *   Checks: every argument check (NULL pointers, alignment, sizes, a
 *   non-finite scale, the limit below) runs before the set-up and the
 *   memset, so a rejected call touches no device and launches nothing.
 *   Limits: returns PA_ERR_WORKSPACE, launching nothing, when the counters
 *   alone (8 + 4 * num_seqs * num_heads bytes, rounded up to 256) exceed
 *   PA_STATIC_SCRATCH_BYTES.
 *   Concurrency: all calls on a device share the one array, so calls whose
 *   kernels may overlap on the GPU (different streams, or other host threads)
 *   race and corrupt each other's results; serialise them.
 */
int pa_decode_static(void *out, const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_tables, const int32_t *context_lens, float scale,
                     int32_t max_blocks_per_seq, const pa_dims *dims, void *stream);

/*
 * KV block manager (host only; no CUDA call).
 *
 * The bookkeeping half of the paged cache: blocks are handed out one at a
 * time from a free list, ceil(tokens / block_size) per sequence, and running
 * out is an error (doramagic.ai vLLM manual, "KVCacheManager 缓存管理"); each
 * sequence keeps a block table of logical -> physical blocks ("vLLM 2026
 * 推理引擎全解", §2.1); blocks may be shared -- a system prompt's full blocks
 * between requests, or every block between the samples forked from one prompt
 * -- and are counted by reference and freed at zero ("vLLM 2026 推理引擎全解",
 * §2.3; mjmagnets.cn vLLM tutorial, §2.1; doramagic.ai vLLM manual, "共享机制").
 * An append that would write into a block another sequence still references
 * first takes a fresh block and reports a (source, destination) pair to copy
 * with pa_copy_blocks (copy-on-write).
 *
 * Sequence ids are small non-negative integers, reused after pa_kvm_free.
 * Calls return a pa_status (PA_ERR_OUT_OF_BLOCKS when the free list is
 * empty, leaving the manager unchanged) unless stated.  Not thread-safe.
 */
typedef struct pa_kv_manager pa_kv_manager;

/* A manager of blocks 0 .. num_blocks-1.  shuffle_seed != 0 shuffles the
 * free list with a seeded Fisher-Yates (splitmix64); 0 keeps 0, 1, 2, ...
 * Returns NULL on invalid sizes or out of host memory. */
pa_kv_manager *pa_kvm_create(int32_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq,
                             uint64_t shuffle_seed);
void pa_kvm_destroy(pa_kv_manager *m);
/* Free blocks (-1 for a NULL manager). */
int32_t pa_kvm_num_free_blocks(const pa_kv_manager *m);
/* Reference count of a block (-1 if out of range). */
int32_t pa_kvm_refcount(const pa_kv_manager *m, int32_t block);
/* A new sequence holding num_tokens tokens.  With parent >= 0, its first
 * shared_blocks blocks are the parent's (they must be full in the parent and
 * lie within num_tokens); the rest are fresh.  With parent < 0,
 * shared_blocks must be 0. */
int pa_kvm_add_sequence(pa_kv_manager *m, int32_t num_tokens, int32_t parent,
                        int32_t shared_blocks, int32_t *seq_out);
/* A new sequence sharing every block of parent, a partial last one included. */
int pa_kvm_fork(pa_kv_manager *m, int32_t parent, int32_t *seq_out);
/* Extend seq by one token: *slot_out = its slot (block * block_size + offset).
 * If that token lands in a block another sequence references, the block is
 * replaced by a fresh one and *copy_src_out / *copy_dst_out name the copy to
 * make before writing the token; otherwise both are -1. */
int pa_kvm_append(pa_kv_manager *m, int32_t seq, int32_t *slot_out, int32_t *copy_src_out,
                  int32_t *copy_dst_out);
/* Release a sequence and its block references. */
int pa_kvm_free(pa_kv_manager *m, int32_t seq);
/* Tokens of seq (-1 if unknown). */
int32_t pa_kvm_context_len(const pa_kv_manager *m, int32_t seq);
/* Slot of token `token` of seq. */
int pa_kvm_slot(const pa_kv_manager *m, int32_t seq, int32_t token, int32_t *slot_out);
/* Batch rows: for each seqs[i] (host), row i of tables_out [num_seqs, row_len]
 * gets the block table padded with -1 and context_lens_out[i] its length; a
 * negative seqs[i] gives an empty row of length 0 (batch padding). */
int pa_kvm_block_tables(const pa_kv_manager *m, const int32_t *seqs, int32_t num_seqs,
                        int32_t *tables_out, int32_t row_len, int32_t *context_lens_out);

/* Groups for pa_decode_shared_prefix from the manager's sharing records, for
 * the batch rows seqs[0 .. num_seqs) in that order (negative ids are padding
 * rows).  Consecutive rows form a group when their tables start with the same
 * physical blocks: the group's prefix is what its first two rows share, and
 * every later member shares at least that much with the first row.  Only
 * blocks that are full in every member count (a block still being filled,
 * shared after a fork, is left to each member's suffix).  Rows that share
 * nothing with the next row are gathered into groups of prefix 0.  Every row
 * belongs to exactly one group.  Writes group_start_out[num_groups + 1] and
 * group_prefix_out[num_groups] (host arrays of max_groups + 1 and max_groups
 * entries); PA_ERR_SHAPE if more than max_groups groups are needed or an id
 * is unknown.  Sharers must be adjacent in the batch to be grouped. */
int pa_kvm_prefix_groups(const pa_kv_manager *m, const int32_t *seqs, int32_t num_seqs,
                         int32_t *group_start_out, int32_t *group_prefix_out, int32_t max_groups,
                         int32_t *num_groups_out);

/*
 * Wait for `stream`, then return (in *flags, host) and clear the current
 * device's error word: an OR of PA_DEVERR_* bits set by kernels since the last
 * read.  The word is shared by all streams of the device.
 */
int pa_device_errors(void *stream, uint32_t *flags);

/*
 * pa_selftest_wait_timeout -- check, on the current device, the bounded waits
 * that every kernel of the library relies on (the pages have no counterpart:
 * this is failure detection for the library itself).  Launches one CTA on
 * `stream` that waits on an mbarrier phase nothing completes, then on a
 * shared-memory word nothing sets, then drains; each wait must give up after
 * its limit (about 1 s each, so the call takes about 3 s) and record
 * PA_DEVERR_TIMEOUT.  Synchronises the stream.  results (host, int[3]) gets
 * 1 for each wait that (wrongly) succeeded, 0 for each that gave up.  The
 * error word is left set for pa_device_errors to read.  Returns PA_OK or
 * PA_ERR_CUDA.
 */
int pa_selftest_wait_timeout(int32_t *results, void *stream);

/* Human-readable name of a pa_status value. */
const char *pa_status_string(int status);

/* cudaError_t of the most recent PA_ERR_CUDA on this host thread. */
int pa_last_cuda_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
