/*
 * pagedkv.h -- C ABI of the paged KV-cache attention library (libpagedkv.so).
 *
 * One GPU (sm_103a).  The library allocates no device memory: the caller owns
 * every buffer and passes device pointers.  Every compute call is asynchronous
 * on the given CUDA stream (a cudaStream_t passed as void*; NULL is the legacy
 * default stream), never synchronises, and never throws.  Arguments are
 * validated on the host before anything is launched; a rejected call launches
 * nothing and returns a negative pkv_status.
 *
 * Data model (sources: openeuler.csdn.net PagedAttention notes, "vLLM -
 * PagedAttention", "Block Table 数据结构" and "Attention 计算时的 Block 映射
 * （CUDA Kernel 伪代码）"; "第32讲 … Prefill vs Decode …", §3.4 GQA):
 *   - the K cache and the V cache are each laid out
 *       [num_blocks][num_kv_heads][block_size][head_dim]
 *     so one (block, KV head) tile of block_size rows is contiguous;
 *   - block_size is 16 tokens;
 *   - block_tables is [num_seqs][max_blocks_per_seq] int32, row-major: entry j
 *     of row s is the physical block holding tokens 16j .. 16j+15 of sequence s.
 *     Entries past ceil(context_lens[s] / 16) are never read;
 *   - a slot is physical_block * block_size + offset;
 *   - query head h reads KV head h / (num_heads / num_kv_heads) (consecutive
 *     groups);
 *   - context_lens[s] counts every token of sequence s, including the new ones
 *     whose K/V pkv_reshape_and_cache has already written;
 *   - q and out are [rows][num_heads][head_dim] contiguous, in q_dtype.
 *
 * Supported: head_dim 64 or 128; block_size 16; num_heads a multiple of
 * num_kv_heads with num_heads / num_kv_heads <= 16; q_dtype F16 or BF16;
 * the cache dtype equal to q_dtype or FP8_E4M3.  Device pointers to caches,
 * q, k, v and out must be 16-byte aligned.
 *
 * Device-side checks.  Each compute call takes `device_errors`, a device
 * pointer to one uint32_t owned by the caller (or NULL to skip reporting).
 * Kernels OR PKV_DEVERR_* bits into it when they meet a block id outside the
 * pool, a context length beyond the table or the launch bounds, a slot outside
 * the pool, or a device-side wait that gave up.  Such data is never read or
 * written out of bounds: the offending access is clamped or skipped and the
 * result of that row is unspecified.  pkv_check_errors reads and clears it.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PKV_F16 = 0, PKV_BF16 = 1, PKV_FP8_E4M3 = 2 } pkv_dtype;

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = -1, /* a null pointer, a bad size, a misaligned pointer */
  PKV_ERR_UNSUPPORTED = -2, /* a valid but unsupported shape or dtype combination */
  PKV_ERR_WORKSPACE = -3,   /* workspace missing or smaller than the size function says */
  PKV_ERR_CUDA = -4,        /* the CUDA runtime reported an error at launch */
  PKV_ERR_DEVICE = -5,      /* pkv_check_errors: a device-side check failed */
  PKV_ERR_TIMEOUT = -6,     /* pkv_check_errors: a device-side wait gave up */
  PKV_ERR_NO_BLOCKS = -7    /* the block pool holds fewer free blocks than the call needs */
} pkv_status;

#define PKV_DEVERR_BLOCK_ID 0x1u    /* block table entry outside [0, num_blocks) */
#define PKV_DEVERR_CONTEXT 0x2u     /* context/query length beyond the table or launch bounds */
#define PKV_DEVERR_SLOT 0x4u        /* slot_mapping entry >= num_blocks * block_size */
#define PKV_DEVERR_TIMEOUT 0x8u     /* a wait on an asynchronous copy or MMA gave up */

/*
 * Scatter new keys and values into the paged caches through a slot mapping.
 * Source: devpress.csdn.net vLLM overview, "8、推理流程" (each layer's K and V
 * are stored into the paged cache before attention reads it);
 * openeuler.csdn.net PagedAttention notes, "Block Table 数据结构"
 * (slot = physical_block * block_size + offset).
 *
 *   k, v          [num_tokens][num_kv_heads][head_dim], src_dtype (F16/BF16)
 *   k_cache,
 *   v_cache       caches as above, cache_dtype
 *   slot_mapping  [num_tokens] int64; token t goes to slot slot_mapping[t].
 *                 Negative entries are padding and are skipped.  Entries
 *                 >= num_blocks * block_size are skipped and flagged
 *                 PKV_DEVERR_SLOT.  Two tokens with one slot is a caller
 *                 error (which one lands is unspecified).
 *   cache_dtype   == src_dtype: the element bits are copied.
 *                 FP8_E4M3: each element becomes E4M3(x / scale) with an IEEE
 *                 float division, round to nearest even, saturating to +-448;
 *                 scale is k_scale for K and v_scale for V (per tensor).
 * num_tokens == 0 launches nothing and returns PKV_OK.
 */
int pkv_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                          const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                          int head_dim, int block_size, int num_blocks, pkv_dtype src_dtype,
                          pkv_dtype cache_dtype, float k_scale, float v_scale,
                          uint32_t* device_errors, void* stream);

/*
 * Bytes of device workspace pkv_paged_attention_decode needs for these
 * arguments (0 when the context fits one partition).  partition_size 0 means
 * the library's choice (the value the decode call would use).
 */
size_t pkv_decode_workspace_size(int num_seqs, int num_heads, int head_dim,
                                 int max_context_len, int partition_size);

/*
 * Decode attention: one query token per sequence attends every token of its
 * context through the block table.
 * Sources: "第32讲 … Prefill vs Decode …", §3.1 (softmax(q K^T / sqrt(d_k)) V
 * over the cached K_{1:t}, V_{1:t}); openeuler.csdn.net PagedAttention notes,
 * "Attention 计算时的 Block 映射（CUDA Kernel 伪代码）" (block_idx = i / 16,
 * offset = i % 16, physical_block = block_table[block_idx]);
 * devpress.csdn.net vLLM overview, "3、PagedAttention (3)" (per-block partial
 * results combined) and "9、FlashAttention (4)" (running max and sum of
 * exponentials, rescaled).
 *
 *   out   [num_seqs][num_heads][head_dim], q_dtype; row s, head h is
 *         sum_t softmax_t(scale * q[s,h] . K[s,t]) V[s,t] over
 *         t < context_lens[s]; a sequence with context 0 gets zeros.
 *   q     [num_seqs][num_heads][head_dim], q_dtype
 *   kv_dtype FP8_E4M3: K and V elements are decode(byte) * k_scale / v_scale;
 *         otherwise the scales are ignored.
 *   max_context_len  an upper bound of context_lens (sizes the launch; no
 *         device-to-host read).  Longer contexts are flagged PKV_DEVERR_CONTEXT.
 *   partition_size   tokens per split of the context (multiple of 16, at
 *         most 512); 0 = the library's choice.  Contexts longer than one
 *         partition are computed per partition into the workspace and
 *         combined by a log-sum-exp merge.
 *   workspace, workspace_bytes  device scratch of at least
 *         pkv_decode_workspace_size(...) bytes, 256-byte aligned; may be NULL
 *         when that size is 0.  Its contents need no initialisation.
 */
int pkv_paged_attention_decode(void* out, const void* q, const void* k_cache,
                               const void* v_cache, const int32_t* block_tables,
                               const int32_t* context_lens, int num_seqs, int num_heads,
                               int num_kv_heads, int head_dim, int block_size,
                               int max_blocks_per_seq, int num_blocks, int max_context_len,
                               float scale, pkv_dtype q_dtype, pkv_dtype kv_dtype,
                               float k_scale, float v_scale, int partition_size,
                               void* workspace, size_t workspace_bytes,
                               uint32_t* device_errors, void* stream);

/*
 * Decode attention that allocates nothing and takes no workspace.
 * (The source pages have no counterpart: this entry point exists for callers
 * of the library, not for the method.)
 *
 * For callers that cannot call cudaMalloc or hand over scratch memory: for
 * example a host framework that owns all device memory through its own pool
 * and forbids plugins from allocating, or a latency-critical loop that must
 * not pay the implicit synchronisation of cudaMalloc/cudaFree.  It computes
 * exactly what pkv_paged_attention_decode computes, with the same arguments
 * minus the workspace, and keeps the split-K scratch in one fixed device
 * array of PKV_DECODE_NOALLOC_SCRATCH_BYTES inside the library.
 *
 *   - The array is reserved on every GPU where this entry point is used and
 *     stays reserved until the process exits.
 *   - The array used is the one on the CURRENT device (cudaGetDevice): make
 *     the device that holds the tensors current before the call.  The first
 *     call on a device looks up the array's address (with that device
 *     current); make that first call before any stream capture.
 *   - Calls whose pkv_decode_workspace_size(...) exceeds
 *     PKV_DECODE_NOALLOC_SCRATCH_BYTES are rejected with PKV_ERR_WORKSPACE
 *     before anything is launched.
 *   - All calls on a device share the one array, and it keeps the previous
 *     call's contents.  Every byte a call reads is written earlier in that same
 *     call, so nothing needs clearing.  Calls that overlap on the GPU (on
 *     different streams, without ordering between them) race on the array and
 *     give undefined results.
 *   - No cudaMalloc, cudaFree or allocating library routine is called.
 */
#define PKV_DECODE_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int pkv_paged_attention_decode_noalloc(void* out, const void* q, const void* k_cache,
                                       const void* v_cache, const int32_t* block_tables,
                                       const int32_t* context_lens, int num_seqs,
                                       int num_heads, int num_kv_heads, int head_dim,
                                       int block_size, int max_blocks_per_seq, int num_blocks,
                                       int max_context_len, float scale, pkv_dtype q_dtype,
                                       pkv_dtype kv_dtype, float k_scale, float v_scale,
                                       int partition_size, uint32_t* device_errors,
                                       void* stream);

/*
 * Bytes of device workspace pkv_paged_attention_prefill_chunk needs (256-byte
 * aligned when passed): the larger of the CUDA-core path's split-K partials
 * and, for head_dim 128, the tensor-core path's split query of an E4M3-cache
 * call (two E4M3 bytes and one fp32 scale per query row and head).
 */
size_t pkv_prefill_workspace_size(int total_q, int num_heads, int head_dim,
                                  int max_context_len, int max_q_len);

/*
 * Chunked-prefill attention: each sequence contributes its last q_len tokens
 * as queries (a chunk of a prompt, or a single decode token), and each of
 * them attends causally to the paged context before it and to itself.
 * Sources: "第32讲 … Prefill vs Decode …", §5.4 (prompts cut into chunks of
 * e.g. 512 tokens, each chunk attending the prior context); devpress.csdn.net
 * vLLM overview, "9、FlashAttention (3)" (query blocks x key/value blocks).
 *
 *   q, out           [total_q][num_heads][head_dim], q_dtype
 *   query_start_loc  [num_seqs + 1] int32, non-decreasing, [0] = 0,
 *                    [num_seqs] = total_q; sequence s owns query rows
 *                    query_start_loc[s] .. query_start_loc[s+1]-1.
 *   The query at row query_start_loc[s] + i sits at absolute position
 *   pos = context_lens[s] - q_len_s + i and attends keys 0..pos.
 *   max_q_len        an upper bound of every q_len_s (sizes the launch).
 *   workspace        at least pkv_prefill_workspace_size(...) bytes, 256-byte
 *                    aligned; may be NULL for 16-bit caches at head_dim 128
 *                    with num_heads / num_kv_heads dividing 128 (the
 *                    tensor-core kernel), which need none.  E4M3 caches on
 *                    that kernel split the query into it (PKV_ERR_WORKSPACE
 *                    when it is missing or short).
 *   Other arguments as for pkv_paged_attention_decode.
 */
int pkv_paged_attention_prefill_chunk(void* out, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_tables,
                                      const int32_t* context_lens,
                                      const int32_t* query_start_loc, int num_seqs,
                                      int total_q, int max_q_len, int num_heads,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int max_blocks_per_seq, int num_blocks,
                                      int max_context_len, float scale, pkv_dtype q_dtype,
                                      pkv_dtype kv_dtype, float k_scale, float v_scale,
                                      void* workspace, size_t workspace_bytes,
                                      uint32_t* device_errors, void* stream);

/*
 * Draft-tree verification: chunked-prefill attention in which each sequence's
 * chunk is a tree of at most 64 draft tokens (speculative decoding, verified
 * in one pass), and each draft token sees the context before the chunk plus
 * only its own ancestors and itself.
 * Sources: openeuler.csdn.net PagedAttention notes, "MEDUSA推理框架",
 * "Tree Attention：" (candidate tokens of several heads form a tree verified
 * under one attention mask) and "EAGLE2推理", "重排阶段" (the mask lets each
 * token see only its ancestors).
 *
 *   tree_mask  [total_q] uint64: for the query at row query_start_loc[s] + i,
 *              bit j set = the chunk's token j (position context_lens[s] -
 *              q_len_s + j) is visible to it.  Bits 0..i for every i give
 *              ordinary causal chunk attention.  Bits past the chunk are ignored.
 *   max_q_len  at most 64 (PKV_ERR_INVALID_ARG otherwise); a longer chunk
 *              found on the device is cut to 64 queries and flagged
 *              PKV_DEVERR_CONTEXT.
 *   Supported: 16-bit caches (kv_dtype == q_dtype), head_dim 128, query heads
 *   per KV head dividing 128, at most 1024 sequences; otherwise
 *   PKV_ERR_UNSUPPORTED.  No workspace.  Other arguments as for
 *   pkv_paged_attention_prefill_chunk.
 */
int pkv_paged_attention_prefill_tree(void* out, const void* q, const void* k_cache,
                                     const void* v_cache, const int32_t* block_tables,
                                     const int32_t* context_lens, const int32_t* query_start_loc,
                                     const uint64_t* tree_mask, int num_seqs, int total_q,
                                     int max_q_len, int num_heads, int num_kv_heads, int head_dim,
                                     int block_size, int max_blocks_per_seq, int num_blocks,
                                     int max_context_len, float scale, pkv_dtype q_dtype,
                                     pkv_dtype kv_dtype, float k_scale, float v_scale,
                                     uint32_t* device_errors, void* stream);

/*
 * Bytes of device workspace pkv_paged_attention_decode_cascade needs.
 */
size_t pkv_cascade_workspace_size(int num_seqs, int num_heads, int head_dim,
                                  int max_context_len, int max_prefix_len);

/*
 * Cascade (shared-prefix) decode: the same result as pkv_paged_attention_decode,
 * for a batch in which groups of sequences share a prompt's blocks by
 * reference (parallel samples of one prompt).  Each shared block is read once
 * per group instead of once per sequence: every member's query attends the
 * shared prefix in one pass, each sequence attends its own keys in a second,
 * and the partial results are combined by a log-sum-exp merge.
 * Sources: openeuler.csdn.net PagedAttention notes, "vLLM - PagedAttention",
 * "机制 2：写时复制（Copy-on-Write）" (parallel samples of one prompt share its
 * physical blocks with a reference count, private blocks only from the
 * diverging point); devpress.csdn.net vLLM overview, "9、FlashAttention (4)"
 * (partial results over disjoint key sets combined by running max and sum of
 * exponentials).
 *
 *   group_start  [num_groups + 1] int32: group g is the sequences
 *         group_start[g] .. group_start[g+1]-1 (consecutive; [0] = 0,
 *         [num_groups] = num_seqs, non-decreasing).
 *   prefix_lens  [num_seqs] int32: the shared prefix of each sequence, in
 *         tokens: a multiple of 16, at most its context, equal for the
 *         members of a group, whose block tables agree on those blocks (the
 *         prefix is read through the group's first member).  0 = nothing
 *         shared.  A length that is not whole blocks or exceeds the context is
 *         cut back and flagged PKV_DEVERR_CONTEXT.
 *   max_prefix_len  an upper bound of prefix_lens (sizes the workspace).
 *   workspace  at least pkv_cascade_workspace_size(...) bytes, 256-byte
 *         aligned; never NULL for num_seqs > 0.
 *   Supported: 16-bit caches (kv_dtype == q_dtype), head_dim 128, 2..16 query
 *   heads per KV head dividing 128, at most 1024 groups; otherwise
 *   PKV_ERR_UNSUPPORTED.  Other arguments as for pkv_paged_attention_decode.
 */
int pkv_paged_attention_decode_cascade(void* out, const void* q, const void* k_cache,
                                       const void* v_cache, const int32_t* block_tables,
                                       const int32_t* context_lens, const int32_t* group_start,
                                       const int32_t* prefix_lens, int num_seqs, int num_groups,
                                       int num_heads, int num_kv_heads, int head_dim,
                                       int block_size, int max_blocks_per_seq, int num_blocks,
                                       int max_context_len, int max_prefix_len, float scale,
                                       pkv_dtype q_dtype, pkv_dtype kv_dtype, float k_scale,
                                       float v_scale, void* workspace, size_t workspace_bytes,
                                       uint32_t* device_errors, void* stream);

/*
 * A mixed batch in one launch: the step's single-token decode rows and its
 * prefill chunks ("第32讲 … Prefill vs Decode …", §5.4 chunked prefill: one
 * batch carries the running decodes and slices of new prompts).  The result
 * equals pkv_paged_attention_decode on the decode rows plus
 * pkv_paged_attention_prefill_chunk on the chunks; with 16-bit caches,
 * head_dim 128 and num_heads / num_kv_heads in 2..8, one kernel does both
 * (its CTAs split between the two kinds of work), followed by the
 * partition merge of the decode rows when their contexts exceed 512 tokens.
 * Other shapes run the two calls one after the other.
 *
 *   sequences     [0, num_decode) are decode rows: query row s, and
 *                 query_start_loc[s] = s for s <= num_decode;
 *                 [num_decode, num_seqs) are chunks with query rows
 *                 query_start_loc[s] .. query_start_loc[s + 1] - 1.
 *   block_tables,
 *   context_lens  one row / entry per sequence, in the same order.
 *   max_context_len  bounds every context_lens entry; max_q_len the chunks.
 *   prefill_ctas  0: the kernel divides the SMs between chunks and decode
 *                 rows from their lengths; > 0: the chunks get that many CTAs
 *                 (clamped to [1, SMs - 1]).
 *   workspace     at least pkv_mixed_workspace_size bytes, 256-byte aligned
 *                 (NULL when that is 0).
 * Other arguments as for pkv_paged_attention_prefill_chunk.
 */
size_t pkv_mixed_workspace_size(int num_decode, int total_q, int num_heads, int head_dim,
                                int max_context_len);
int pkv_paged_attention_mixed(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, const int32_t* context_lens,
                              const int32_t* query_start_loc, int num_decode, int num_seqs,
                              int total_q, int max_q_len, int num_heads, int num_kv_heads,
                              int head_dim, int block_size, int max_blocks_per_seq,
                              int num_blocks, int max_context_len, float scale,
                              pkv_dtype q_dtype, pkv_dtype kv_dtype, float k_scale,
                              float v_scale, int prefill_ctas, void* workspace,
                              size_t workspace_bytes, uint32_t* device_errors, void* stream);

/*
 * Whole-block copies in both caches: the device half of copy-on-write
 * (openeuler.csdn.net PagedAttention notes, "机制 2：写时复制": a request that
 * writes into a block it shares first gets its own copy).
 *
 *   block_pairs  device [num_pairs][2] int32: (source, destination) block ids.
 *                Destinations must be distinct and must not be sources of the
 *                same call (the pairs run concurrently).  A pair with an id
 *                outside [0, num_blocks) is skipped and flagged
 *                PKV_DEVERR_BLOCK_ID.
 *   caches       as for pkv_reshape_and_cache, cache_dtype F16, BF16 or
 *                FP8_E4M3; every (K and V) byte of the destination block
 *                becomes the source block's.
 * num_pairs == 0 launches nothing and returns PKV_OK.
 */
int pkv_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_pairs, int num_pairs,
                    int num_kv_heads, int head_dim, int block_size, int num_blocks,
                    pkv_dtype cache_dtype, uint32_t* device_errors, void* stream);

/*
 * Host block pool with prefix caching.  Sources: "第34讲 … vLLM 生产级系统架构
 * 全景剖析与四重加速引擎", §1.2 (KVCacheManager.allocate_slots / free, BlockPool,
 * FreeKVCacheBlockQueue), §2.2 (longest-prefix reuse with ref_cnt), §2.3
 * (cached free blocks, LRU eviction); openeuler.csdn.net PagedAttention notes,
 * "机制 2：写时复制" (fork, copy-on-write).
 *
 * Host memory only, no CUDA calls; not thread-safe (serialise calls on one
 * pool and its requests).  The pool owns its requests' bookkeeping; a request
 * must be freed before its pool is destroyed.
 *
 * Semantics:
 *   - a fresh pool's free queue holds blocks 0, 1, ..., num_blocks - 1;
 *     allocation takes the queue's head; a block whose reference count drops
 *     to 0 joins the tail (a request releases its blocks last block first);
 *   - a block is cached when it becomes full: it is registered under its
 *     token prefix (every token from the request's start through the block's
 *     last), unless that prefix is already registered to another block.  A
 *     cached block keeps its registration at count 0 and is dropped from the
 *     cache (evicted) only when allocation takes it from the queue;
 *   - pkv_request_match_prefix reuses the longest run of cached blocks that
 *     spells the start of the prompt, stopping before the block that holds
 *     the prompt's last token (one token is always left to compute).
 *     Reused blocks gain a reference and leave the free queue;
 *   - pkv_request_append fills the last block first and takes new blocks
 *     from the head.  If the last block is partial and shared (after a fork),
 *     a private copy is made first: cow_out receives {source, copy} and the
 *     caller copies the cache bytes (pkv_copy_blocks) before writing the new
 *     tokens' K/V.  All or nothing: PKV_ERR_NO_BLOCKS leaves the pool and the
 *     request unchanged.
 */
typedef struct pkv_block_pool pkv_block_pool;
typedef struct pkv_request pkv_request;

/* *out receives a new pool (NULL on error).  num_blocks >= 0, block_size > 0. */
int pkv_block_pool_create(int32_t num_blocks, int32_t block_size, pkv_block_pool** out);
void pkv_block_pool_destroy(pkv_block_pool* pool);
/* Blocks in the free queue (cached or not); -1 for a NULL pool. */
int32_t pkv_block_pool_num_free(const pkv_block_pool* pool);
/* Registered (cached) blocks, in use or free; -1 for a NULL pool. */
int32_t pkv_block_pool_num_cached(const pkv_block_pool* pool);
/* Reference count / 1 if cached else 0; -1 for a bad pool or block id. */
int32_t pkv_block_pool_ref_cnt(const pkv_block_pool* pool, int32_t block);
int32_t pkv_block_pool_is_cached(const pkv_block_pool* pool, int32_t block);
/* Copies up to max ids of the free queue, head first, into out (may be NULL
 * when max is 0); returns the queue's length. */
int32_t pkv_block_pool_queue(const pkv_block_pool* pool, int32_t* out, int32_t max);

/* *out receives a new, empty request of the pool. */
int pkv_request_create(pkv_block_pool* pool, pkv_request** out);
/* On an empty request only (PKV_ERR_INVALID_ARG otherwise): reuse the cached
 * prefix of tokens[0 .. num_tokens); *matched_out (may be NULL) receives the
 * tokens covered, a multiple of block_size.  The caller then appends
 * tokens[matched ..]. */
int pkv_request_match_prefix(pkv_request* req, const int32_t* tokens, int32_t num_tokens,
                             int32_t* matched_out);
/* Appends num_tokens token ids.  slots_out (may be NULL) receives each new
 * token's slot, physical_block * block_size + offset, for pkv_reshape_and_cache;
 * cow_out (may be NULL) receives {source, copy} or {-1, -1}. */
int pkv_request_append(pkv_request* req, const int32_t* token_ids, int32_t num_tokens,
                       int64_t* slots_out, int32_t* cow_out);
/* *out receives a request sharing every block of req (each gains a reference). */
int pkv_request_fork(const pkv_request* req, pkv_request** out);
/* Releases the request's blocks, last block first, and frees it. NULL is a no-op. */
void pkv_request_free(pkv_request* req);
/* Tokens held; -1 for NULL. */
int32_t pkv_request_num_tokens(const pkv_request* req);
/* Copies up to max block ids; returns the request's block count (-1 for NULL). */
int32_t pkv_request_block_table(const pkv_request* req, int32_t* out, int32_t max);
/* Host [num_reqs][max_blocks] block tables (entries past a request's blocks
 * are 0) and context_lens (may be NULL) for a batch of requests, in the layout
 * the attention calls take.  PKV_ERR_INVALID_ARG (nothing written) when a
 * request holds more than max_blocks blocks. */
int pkv_requests_block_tables(const pkv_request* const* reqs, int32_t num_reqs,
                              int32_t max_blocks, int32_t* block_tables, int32_t* context_lens);

/*
 * Synchronises `stream`, reads the device error word, clears it, and returns
 * PKV_OK, PKV_ERR_TIMEOUT (a wait gave up) or PKV_ERR_DEVICE (any other bit);
 * PKV_ERR_CUDA if the stream reports an error.  *bits_out (may be NULL)
 * receives the raw bits.
 */
int pkv_check_errors(uint32_t* device_errors, uint32_t* bits_out, void* stream);

/*
 * Test hook for the failure detection above (the pages have no counterpart:
 * "第34讲 …", §1.2 speaks of preemption and service levels only).  Arms the
 * next attention call made in this process (decode, prefill chunk, draft
 * tree, mixed batch or cascade): in that call's tensor-core kernel(s) the
 * first copy producer of the first CTA does not issue its skip_copy-th tile
 * copy
 * (counted from 1), and every device-side wait is bounded by wait_limit_us
 * microseconds (0: the default of about 2 s) instead of the default.  The
 * waits for the missing tile then run out: the kernel ORs
 * PKV_DEVERR_TIMEOUT into device_errors, lets its issued copies and MMAs
 * finish, releases its tensor memory and returns, and pkv_check_errors then
 * returns PKV_ERR_TIMEOUT.  The rows of that CTA's work are unspecified;
 * later calls are unaffected.  A call that runs on the CUDA-core decode
 * kernel (one query head per KV head, or head_dim 64) takes the hook without
 * effect: that kernel carries no hook code in its copy loop.  No copy in flight is ever abandoned and no
 * GPU fault is raised.  The hook is taken by exactly one call.
 * PKV_ERR_INVALID_ARG when skip_copy <= 0.
 */
int pkv_debug_arm_wait_timeout(int skip_copy, unsigned wait_limit_us);

/*
 * Selects the kernel that runs causal chunks (pkv_paged_attention_prefill_chunk)
 * and draft trees (pkv_paged_attention_prefill_tree) on tensor cores:
 *   1  pairs of CTAs that share each 256-row query tile (each CTA loads half of
 *      every K/V tile);
 *   0  one CTA per 128-row tile;
 *   2  (the default) pairs for draft trees, one CTA per tile for causal chunks.
 * All compute the same attention, bit for bit; the switch exists to test and
 * measure one against the other.  Process-wide; returns the previous setting,
 * or PKV_ERR_INVALID_ARG for another value.
 */
int pkv_debug_prefill_pairs(int mode);

/* A static, human-readable name for a pkv_status value. */
const char* pkv_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
