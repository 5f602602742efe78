/*
 * pagedkv.h -- C ABI of libpagedkv.so: the paged KV-cache decode path on one GB300.
 *
 * The operations follow the statement of the problem on the pages:
 *  - the KV cache is cut into fixed-size blocks of 16 tokens handed out from one pool,
 *    and each request's block table maps its logical block i to a physical block
 *    ("Continuous batching and PagedAttention", section 3 PagedAttention;
 *    "System-level optimization: batching, PagedAttention and FlashAttention",
 *    section 2.3 PagedAttention solution);
 *  - each decode step computes only the new token's K/V and appends it to the cache
 *    ("Inference optimization", section "KV cache");
 *  - shared blocks are copied when a request diverges (copy-on-write, "Continuous
 *    batching and PagedAttention", section 3, copy-on-write sharing);
 *  - attention is softmax(q K^T * scale) V with scale = head_dim^-1/2
 *    ("System-level optimization", sections 3.1 and 3.3).
 *
 * Conventions shared by every call
 *  - bf16 tensors are passed as uint16_t bit patterns, row-major:
 *      q, out              [num_seqs][num_q_heads][head_dim]
 *      k_cache, v_cache    [num_blocks][num_kv_heads][block_size][head_dim]
 *      k_new, v_new        [num_tokens][num_kv_heads][head_dim]
 *    int32 block_tables [num_seqs][max_blocks_per_seq], int32 context_lens [num_seqs],
 *    int64 slot_mapping [num_tokens], int32 block_pairs [num_pairs][2] = (src, dst).
 *  - Every pointer argument of the GPU calls is a device pointer owned by the caller.
 *    The library never allocates, frees or synchronises on these calls; work is
 *    enqueued on `stream` (a cudaStream_t; NULL is the legacy default stream).
 *  - Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *  - context_lens counts every token attended, the one written this step included.
 *  - Token t of sequence s lives in block block_tables[s][t / 16] at offset t % 16;
 *    slot = physical_block * 16 + offset.
 *  - Return value: PKV_OK, or a negative PKV_ERR_* code for arguments rejected on the
 *    host (nothing is enqueued then), or PKV_ERR_CUDA if a launch failed.
 *  - err_flag (device int32, caller-owned, may be NULL): a kernel that meets a bad
 *    index (block id outside [0, num_blocks), slot outside the pool, context longer
 *    than the block table or than max_context_len) ORs a PKV_DEV_* bit into it and
 *    skips that access.  No kernel traps or waits without a bound.
 *  - head_dim must be 64 or 128; block_size must be 16; q, out, the caches and the
 *    new K/V must be 16-byte aligned.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_OK 0
#define PKV_ERR_NULL (-1)        /* a required pointer is NULL                        */
#define PKV_ERR_SHAPE (-2)       /* a size is out of range or head_dim unsupported    */
#define PKV_ERR_BLOCK_SIZE (-3)  /* block_size is not 16                              */
#define PKV_ERR_ALIGN (-4)       /* a bf16 buffer is not 16-byte aligned              */
#define PKV_ERR_WORKSPACE (-5)   /* workspace smaller than the size query returns     */
#define PKV_ERR_CUDA (-6)        /* a CUDA runtime call or kernel launch failed       */
#define PKV_ERR_OOM (-10)        /* block pool: no free block                         */
#define PKV_ERR_UNKNOWN_SEQ (-11)/* block pool: no such sequence                      */
#define PKV_ERR_DUP_SEQ (-12)    /* block pool: sequence id already in use            */
#define PKV_ERR_REFCOUNT (-13)   /* block pool: refcount underflow (corrupt state)    */
#define PKV_ERR_ARG (-14)        /* block pool: bad argument                          */

#define PKV_DEV_BAD_BLOCK 1      /* block table entry or copy pair outside the pool   */
#define PKV_DEV_BAD_SLOT 2       /* slot_mapping entry >= num_blocks * 16             */
#define PKV_DEV_BAD_CONTEXT 4    /* context_len < 0 or beyond table / max_context_len */
#define PKV_DEV_TIMEOUT 8        /* a bounded wait inside a kernel gave up            */
#define PKV_DEV_LAYOUT 16        /* shared-memory window misaligned (kernel skipped)  */
#define PKV_DEV_BAD_SCALE 32     /* a per-KV-head E4M3 scale is not > 0               */
#define PKV_DEV_BAD_ROW 64       /* a gathered row index outside its table            */

/* Library ABI version: PKV_ABI_VERSION of the build (incremented when an entry point is
 * added or a signature changes).  2 added paged_kv_write_fp8_per_head,
 * paged_attention_decode_fp8_per_head, pkv_pool_save and pkv_pool_load; 3 added
 * paged_decode_step, paged_decode_step_fp8 and pkv_sched_pack; 4 added
 * paged_gather_rows, pkv_step_launch and pkv_engine_step. */
#define PKV_ABI_VERSION 4
int paged_kv_version(void);

/* Human-readable text of a PKV_ERR_* code. Never NULL; static storage. */
const char *paged_kv_strerror(int code);

/*
 * paged_kv_write -- append this step's new tokens to the paged cache.
 * For t < num_tokens and every KV head h:
 *   k_cache[slot/16][h][slot%16][:] = k_new[t][h][:]   (same for v), slot = slot_mapping[t].
 * A negative slot is skipped (padding).  Bit-exact byte movement.  Two tokens with the
 * same slot in one call race (the caller must not do that).
 * Source: "Inference optimization", section "KV cache" (only the new token's K/V is
 * computed and appended) and section "Step 1: KV cache" (the update method).
 */
int paged_kv_write(const uint16_t *k_new, const uint16_t *v_new, const int64_t *slot_mapping,
                   int num_tokens, uint16_t *k_cache, uint16_t *v_cache, int num_blocks,
                   int num_kv_heads, int head_dim, int block_size, int32_t *err_flag,
                   void *stream);

/*
 * paged_kv_check_slots -- host-side validation of a slot mapping (HOST memory) before it
 * is used by paged_kv_write: PKV_OK, or PKV_ERR_ARG if a slot is >= num_blocks *
 * block_size or two tokens share a slot (the writes would race).  Negative slots are
 * padding and ignored.  O(n log n); a debugging aid, not part of the step.
 */
int paged_kv_check_slots(const int64_t *slot_mapping, int num_tokens, int num_blocks,
                         int block_size);

/*
 * paged_block_copy -- copy-on-write of whole blocks.
 * For every pair i: k_cache[dst] = k_cache[src] and v_cache[dst] = v_cache[src], all KV
 * heads, bit-exact.  The dsts of one call must be distinct and no dst may be the src of
 * another pair in the same call (the copies run concurrently).
 * Source: "Continuous batching and PagedAttention", section 3 PagedAttention, the
 * copy-on-write paragraph (a shared block is copied only when a request diverges).
 */
int paged_block_copy(uint16_t *k_cache, uint16_t *v_cache, const int32_t *block_pairs,
                     int num_pairs, int num_blocks, int num_kv_heads, int head_dim,
                     int block_size, int32_t *err_flag, void *stream);

/*
 * Bytes of device workspace paged_attention_decode needs for these sizes.
 * partition_size <= 0 (the automatic size) needs the workspace of 512-token partitions.
 */
size_t paged_attention_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                      int max_context_len, int partition_size);

/*
 * paged_attention_decode -- one query token per sequence attends over its paged cache.
 * For every sequence s and query head h, with n = context_lens[s], g = h / (Hq/Hkv):
 *   x_t = scale * q[s][h] . K_s[t][g],   t < n, where K_s[t] is read through block_tables
 *   out[s][h] = sum_t exp(x_t - max x) V_s[t][g] / sum_t exp(x_t - max x)
 * computed in fp32 from bf16 inputs and rounded to bf16.  n == 0 gives zeros.
 * Long contexts are split into partitions of partition_size tokens (a multiple of 16)
 * whose partial results are merged with a log-sum-exp reduction.  partition_size <= 0
 * lets each call choose on the device, from context_lens, the largest candidate size not
 * above (sum of context_lens x KV heads x query sub-groups) / (d x 4 x SMs), i.e. about
 * d partitions' worth of work per resident CTA of the partition kernel (large batches
 * get fewer partitions: fewer items and partial results to merge): on the tensor-core
 * path with 4 or more query heads per KV head d = 3 and the candidates are 512, 768,
 * 1024, 1536, 2048, 3072 and 4096 tokens; otherwise d = 4 and 512, 1024 or 2048.  The
 * result depends on the split only through fp32 rounding.
 * max_context_len is a host-side upper bound of context_lens (it sizes the workspace);
 * a context above it sets PKV_DEV_BAD_CONTEXT and that sequence's output is zeros.
 * workspace (device, >= paged_attention_workspace_size bytes, 256-byte aligned) is
 * scratch owned by the caller; its contents need no initialisation and are
 * overwritten.  Calls that share a workspace must be ordered on one stream.
 * Source: "System-level optimization", section 3.1 (attention equation) and 3.3
 * (scale); "Continuous batching and PagedAttention", section 3 (block tables).
 */
int paged_attention_decode(uint16_t *out, const uint16_t *q, const uint16_t *k_cache,
                           const uint16_t *v_cache, const int32_t *block_tables,
                           const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int num_blocks, float scale, int partition_size, int max_context_len,
                           void *workspace, size_t workspace_bytes, int32_t *err_flag,
                           void *stream);

/*
 * paged_decode_step -- one whole decode step of one layer: copy-on-write, the paged write
 * of the step's new tokens, then decode attention.  The result is exactly that of
 *   paged_block_copy(k_cache, v_cache, block_pairs, num_pairs, ...);
 *   paged_kv_write(k_new, v_new, slot_mapping, num_tokens, k_cache, v_cache, ...);
 *   paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, ...);
 * (every copy before every write, every write before attention), in three launches
 * instead of five: the copies, the writes and the attention plan share the first.
 * Arguments, layouts, ownership and errors are those of the three calls; num_tokens or
 * num_pairs may be 0 (their pointers may then be NULL).  The pair rules of
 * paged_block_copy apply (distinct dsts, no dst that is also a src); a new token may
 * write into a pair's src or dst block (it lands after the copy).  With num_seqs == 0
 * only the copies and the write run.
 * Source: as the three calls ("Continuous batching and PagedAttention", section 3;
 * "Inference optimization", section "KV cache"; "System-level optimization", sections
 * 3.1 and 3.3).
 */
int paged_decode_step(uint16_t *out, const uint16_t *q, uint16_t *k_cache, uint16_t *v_cache,
                      const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                      int max_blocks_per_seq, int num_q_heads, int num_kv_heads, int head_dim,
                      int block_size, int num_blocks, float scale, int partition_size,
                      int max_context_len, const uint16_t *k_new, const uint16_t *v_new,
                      const int64_t *slot_mapping, int num_tokens, const int32_t *block_pairs,
                      int num_pairs, void *workspace, size_t workspace_bytes, int32_t *err_flag,
                      void *stream);

/* ------------------------------------------------------------------------------------
 * E4M3 (FP8) KV cache.  "Continuous batching and PagedAttention", section 4: the
 * kv_cache_dtype="fp8" option doubles the batch a GPU holds; "Inference optimization",
 * exercise 1: quantised KV caches hold proportionally more concurrent requests.
 * Format: OCP E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
 * largest finite 448).  A cache element is one byte, code = E4M3(x / scale) with the
 * division rounded to nearest in fp32 and the conversion rounded to nearest even with
 * finite saturation; it stands for decode(code) * scale.  One scale per cache (k_scale,
 * v_scale, > 0), or one per KV head (the _per_head entry points; the pages leave the
 * granularity open).  Layouts: k_cache [num_blocks][num_kv_heads][16][head_dim] like the
 * bf16 cache; v_cache transposed within each block, [num_blocks][num_kv_heads][head_dim][16]
 * (so the P.V tile reads consecutive tokens).  Both 16-byte aligned.
 * ------------------------------------------------------------------------------------ */

/* Quantise and scatter the step's bf16 K/V into E4M3 caches (otherwise as
 * paged_kv_write).  head_dim a multiple of 16. */
int paged_kv_write_fp8(const uint16_t *k_new, const uint16_t *v_new, const int64_t *slot_mapping,
                       int num_tokens, uint8_t *k_cache, uint8_t *v_cache, int num_blocks,
                       int num_kv_heads, int head_dim, int block_size, float k_scale,
                       float v_scale, int32_t *err_flag, void *stream);

/* paged_kv_write_fp8 with one scale per KV head: head h's K values are divided by
 * k_scales[h] and its V values by v_scales[h].  k_scales, v_scales: device arrays of
 * num_kv_heads fp32 values, each > 0, read by the kernel (so they may be written by
 * earlier work on the stream); NULL returns PKV_ERR_NULL.  A row whose head has a
 * scale that is not > 0 (zero, negative, NaN) is not written and sets
 * PKV_DEV_BAD_SCALE.  The per-cache scheme is the case of equal entries. */
int paged_kv_write_fp8_per_head(const uint16_t *k_new, const uint16_t *v_new,
                                const int64_t *slot_mapping, int num_tokens, uint8_t *k_cache,
                                uint8_t *v_cache, int num_blocks, int num_kv_heads,
                                int head_dim, int block_size, const float *k_scales,
                                const float *v_scales, int32_t *err_flag, void *stream);

/* Copy-on-write of whole blocks of E4M3 caches (as paged_block_copy, bit-exact). */
int paged_block_copy_fp8(uint8_t *k_cache, uint8_t *v_cache, const int32_t *block_pairs,
                         int num_pairs, int num_blocks, int num_kv_heads, int head_dim,
                         int block_size, int32_t *err_flag, void *stream);

/* Decode attention over E4M3 caches: as paged_attention_decode with every K element
 * decode(code) * k_scale and every V element decode(code) * v_scale.  The scores are
 * formed on tensor cores in f16 (E4M3 codes convert to f16 exactly; q is rounded
 * bf16 -> f16, exact for 2^-14 <= |q| <= 65504) with fp32 accumulation; the softmax
 * weights enter the P.V tile as f16.  head_dim 64 or 128 (else PKV_ERR_SHAPE).  The
 * workspace is the one paged_attention_workspace_size gives. */
int paged_attention_decode_fp8(uint16_t *out, const uint16_t *q, const uint8_t *k_cache,
                               const uint8_t *v_cache, const int32_t *block_tables,
                               const int32_t *context_lens, int num_seqs,
                               int max_blocks_per_seq, int num_q_heads, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks, float scale,
                               float k_scale, float v_scale, int partition_size,
                               int max_context_len, void *workspace, size_t workspace_bytes,
                               int32_t *err_flag, void *stream);

/* paged_attention_decode_fp8 over caches written with paged_kv_write_fp8_per_head:
 * every K element of KV head g is decode(code) * k_scales[g] and every V element
 * decode(code) * v_scales[g], so query head h uses the scales of KV head
 * h / (num_q_heads / num_kv_heads).  k_scales, v_scales: device arrays of num_kv_heads
 * fp32 values, each > 0, read by the kernel; NULL returns PKV_ERR_NULL.  A scale that
 * is not > 0 sets PKV_DEV_BAD_SCALE and the rows of the query heads reading that KV
 * head are then unspecified (nothing is read or written out of bounds). */
int paged_attention_decode_fp8_per_head(uint16_t *out, const uint16_t *q, const uint8_t *k_cache,
                                        const uint8_t *v_cache, const int32_t *block_tables,
                                        const int32_t *context_lens, int num_seqs,
                                        int max_blocks_per_seq, int num_q_heads,
                                        int num_kv_heads, int head_dim, int block_size,
                                        int num_blocks, float scale, const float *k_scales,
                                        const float *v_scales, int partition_size,
                                        int max_context_len, void *workspace,
                                        size_t workspace_bytes, int32_t *err_flag, void *stream);

/* paged_decode_step over E4M3 caches: paged_block_copy_fp8, then the quantising write,
 * then E4M3 decode attention, as one call (see paged_decode_step).  Scales: k_scales and
 * v_scales both non-NULL selects one scale per KV head (the _per_head calls' semantics;
 * k_scale and v_scale are then ignored), both NULL one scale per cache (k_scale, v_scale
 * > 0, else PKV_ERR_SHAPE); one NULL and one not returns PKV_ERR_NULL.  head_dim 64 or
 * 128. */
int paged_decode_step_fp8(uint16_t *out, const uint16_t *q, uint8_t *k_cache, uint8_t *v_cache,
                          const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                          int max_blocks_per_seq, int num_q_heads, int num_kv_heads,
                          int head_dim, int block_size, int num_blocks, float scale,
                          float k_scale, float v_scale, const float *k_scales,
                          const float *v_scales, int partition_size, int max_context_len,
                          const uint16_t *k_new, const uint16_t *v_new,
                          const int64_t *slot_mapping, int num_tokens,
                          const int32_t *block_pairs, int num_pairs, void *workspace,
                          size_t workspace_bytes, int32_t *err_flag, void *stream);

/*
 * paged_attention_decode_noalloc -- paged_attention_decode for callers that cannot
 * allocate device memory (no cudaMalloc on their thread, memory owned by another
 * runtime's pool, or a stream being captured by someone else).  The pages have no
 * counterpart; it is a deployment convenience.
 * Same arguments and result as paged_attention_decode, minus the workspace: the
 * split-K scratch is a fixed device array of PKV_NOALLOC_SCRATCH_BYTES inside the
 * library, which every GPU that loads the library keeps until the process exits.
 * Sizes whose paged_attention_workspace_size exceeds it return PKV_ERR_WORKSPACE and
 * enqueue nothing.  The call allocates nothing (no cudaMalloc/cudaFree or allocating
 * library routine).  Its first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call before any
 * stream capture.  The stream must belong to the current device (the array is chosen
 * by the current device): a stream of another device returns PKV_ERR_ARG.  All calls on
 * one device share the array: calls whose kernels overlap on the GPU (other streams,
 * other threads) race, so order them on one stream.  The array keeps the last call's
 * contents; nothing in it needs clearing.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20)
int paged_attention_decode_noalloc(uint16_t *out, const uint16_t *q, const uint16_t *k_cache,
                                   const uint16_t *v_cache, const int32_t *block_tables,
                                   const int32_t *context_lens, int num_seqs,
                                   int max_blocks_per_seq, int num_q_heads, int num_kv_heads,
                                   int head_dim, int block_size, int num_blocks, float scale,
                                   int partition_size, int max_context_len, int32_t *err_flag,
                                   void *stream);

/*
 * paged_attention_prefill -- chunked prefill: several new query tokens per sequence,
 * each attending causally over the sequence's paged cache.
 * Sequence s owns the L = query_start[s+1] - query_start[s] rows query_start[s] ..
 * query_start[s+1]-1 of q and out ([num_tokens][num_q_heads][head_dim] bf16); they are
 * its last L tokens, so row i (0 <= i < L) is the token at position
 * p = context_lens[s] - L + i, and its K/V must already be in the cache (paged_kv_write
 * of the chunk's slots before this call).  For every such row and query head h, with
 * g = h / (Hq/Hkv):
 *   out[row][h] = sum_{t<=p} exp(x_t - max x) V_s[t][g] / sum_{t<=p} exp(x_t - max x),
 *   x_t = scale * q[row][h] . K_s[t][g]
 * computed on tensor cores (bf16 products, fp32 accumulation and softmax; the weights
 * enter the P.V product rounded to bf16) and rounded to bf16.  L == 1 is a decode row.
 * query_start: int32 [num_seqs + 1], device, non-decreasing, query_start[num_seqs] <=
 * num_tokens.  max_query_len: host upper bound of every L (it sizes the launch).
 * A sequence with L > max_query_len, L > context_lens[s], a context longer than its
 * block table or a query_start outside [0, num_tokens] sets PKV_DEV_BAD_CONTEXT and
 * its rows are left unwritten; a bad block id sets PKV_DEV_BAD_BLOCK.  No workspace.
 * head_dim 64 or 128.
 * Sources: "Continuous batching and PagedAttention", section 2 (chunked prefill) and
 * section 3 (block tables); "System-level optimization", section 3.3 (is_causal=True,
 * scale = head_dim^-1/2).
 */
int paged_attention_prefill(uint16_t *out, const uint16_t *q, const uint16_t *k_cache,
                            const uint16_t *v_cache, const int32_t *block_tables,
                            const int32_t *context_lens, const int32_t *query_start,
                            int num_seqs, int num_tokens, int max_blocks_per_seq,
                            int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            int num_blocks, float scale, int max_query_len, int32_t *err_flag,
                            void *stream);

/*
 * Chunked-prefill kernel selection, process-wide (for measurement; default AUTO = the
 * separate-P tcgen05 kernel, for head_dim 64 and 128, the fastest measured on GB300; the
 * others compute the same result and are kept for comparison).
 * Returns the previous value, or PKV_ERR_ARG for an unknown value.
 */
#define PKV_PREFILL_AUTO 0
#define PKV_PREFILL_MMA 1  /* mma.sync tiles, 64 rows per CTA                         */
#define PKV_PREFILL_TC 2   /* tcgen05 tiles with TMEM accumulators, 128 rows per CTA  */
#define PKV_PREFILL_TC_PAIR 3 /* tcgen05, two 128-row tiles per CTA sharing K/V tiles */
#define PKV_PREFILL_TC_2SM 4  /* tcgen05 on SM pairs (M = 256), head_dim 128; else TC  */
#define PKV_PREFILL_TC_SEP 5  /* tcgen05, one S buffer, P and half of Q in own TMEM    */
int paged_attention_prefill_set_variant(int variant);

/*
 * Attention kernel selection, process-wide (for measurement; the default is AUTO).
 * Returns the previous value, or PKV_ERR_ARG for an unknown value.
 */
#define PKV_ATTN_AUTO 0
#define PKV_ATTN_FMA 1   /* CUDA-core dot products and accumulation */
#define PKV_ATTN_MMA 2   /* tensor-core tiles for the query-group contraction */
int paged_attention_set_variant(int variant);

/* ------------------------------------------------------------------------------------
 * Host block manager ("Continuous batching and PagedAttention", section 3; "System-level
 * optimization", section 2.3): one pool of fixed-size blocks, a block table per
 * sequence, reference counts, fork for shared prefixes / parallel sampling, and
 * copy-on-write when a sequence appends into a block it shares.
 * Allocation order: the free pool is a stack that starts as free_order (first element
 * handed out first; NULL = 0, 1, 2, ...); a freed block goes on top.  pkv_seq_free
 * releases a sequence's blocks from its last logical block to its first.
 * Every failing call leaves the pool unchanged.  Not thread-safe: one pool per thread.
 * ------------------------------------------------------------------------------------ */
typedef struct pkv_pool pkv_pool;

int pkv_pool_create(int num_blocks, int block_size, const int32_t *free_order, pkv_pool **out);
void pkv_pool_destroy(pkv_pool *pool);
int pkv_pool_num_free(const pkv_pool *pool);
int pkv_block_refcount(const pkv_pool *pool, int block);  /* <0 on a bad block id */

int pkv_seq_add(pkv_pool *pool, int64_t seq);
int pkv_seq_fork(pkv_pool *pool, int64_t parent, int64_t child);
int pkv_seq_free(pkv_pool *pool, int64_t seq);
int pkv_seq_num_tokens(const pkv_pool *pool, int64_t seq, int *num_tokens);
int pkv_seq_num_blocks(const pkv_pool *pool, int64_t seq, int *num_blocks);

/* Reserve the slot of the sequence's next token.  *cow_src/*cow_dst = -1 unless the
 * token falls in a shared block, in which case the block was replaced by a fresh one
 * and the caller must copy cow_src -> cow_dst (paged_block_copy) before writing. */
int pkv_seq_append_slot(pkv_pool *pool, int64_t seq, int64_t *slot, int32_t *cow_src,
                        int32_t *cow_dst);

/* `count` append_slot calls, all or nothing.  slots[count] and cow_pairs[2*count] may
 * be NULL; *num_cow (may be NULL) receives the number of pairs written. */
int pkv_seq_append_tokens(pkv_pool *pool, int64_t seq, int count, int64_t *slots,
                          int32_t *cow_pairs, int *num_cow);

/* One decode step: one append_slot per listed sequence, in order, all or nothing.
 * slot_mapping[n]; cow_pairs[2*n] receives the copies to make; *num_cow their count. */
int pkv_pool_step(pkv_pool *pool, const int64_t *seqs, int n, int64_t *slot_mapping,
                  int32_t *cow_pairs, int *num_cow);

/* Block tables [n][max_blocks] (unused entries = pad) and context lengths of `seqs`. */
int pkv_pool_export(const pkv_pool *pool, const int64_t *seqs, int n, int max_blocks,
                    int32_t pad, int32_t *block_tables, int32_t *context_lens);

/* Checkpoint / resume of the host allocator (the pages have none; it lets a serving
 * process save its block bookkeeping beside the KV caches and rebuild it).
 * pkv_pool_save: the snapshot's size in bytes; with buf non-NULL and buf_bytes at least
 * that size it also writes the snapshot there (caller-owned memory).  The snapshot holds
 * the free order, every refcount (retains by a prefix cache included) and every
 * sequence's table and length, as little-endian int64 words.  PKV_ERR_NULL for a NULL
 * pool, PKV_ERR_ARG for a buffer too small.
 * pkv_pool_load: a new pool (release it with pkv_pool_destroy) in the saved state; the
 * next calls on it behave exactly as on the saved pool.  PKV_ERR_ARG, and *out = NULL,
 * for bytes that are not a consistent snapshot (wrong size or magic, ids out of range,
 * counts the buffer is too short to hold, a repeated free block, a free block in a
 * table, a table longer than the pool or not matching its token count, a refcount below
 * its table uses); PKV_ERR_OOM if host memory runs out while building.
 * References held outside sequence tables (pkv_block_retain, the prefix cache) are
 * saved as counts only: the snapshot does not record who holds them, so after a load
 * each such holder must be re-registered (a prefix cache rebuilt over the loaded pool)
 * or its references released with pkv_block_release, else those blocks stay allocated. */
int64_t pkv_pool_save(const pkv_pool *pool, void *buf, int64_t buf_bytes);
int pkv_pool_load(const void *buf, int64_t buf_bytes, pkv_pool **out);

/* ------------------------------------------------------------------------------------
 * Block pool: sharing primitives used by the prefix cache.
 * ------------------------------------------------------------------------------------ */
/* A new sequence whose table starts with `num_blocks` allocated blocks (each refcount
 * + 1), holding num_blocks * block_size tokens already. */
int pkv_seq_add_shared(pkv_pool *pool, int64_t seq, const int32_t *blocks, int num_blocks);
/* One more / one fewer holder of an allocated block (a block returns to the pool when
 * its last holder releases it). */
int pkv_block_retain(pkv_pool *pool, int block);
int pkv_block_release(pkv_pool *pool, int block);

/* ------------------------------------------------------------------------------------
 * Prefix cache: a trie of full prompt blocks with LRU eviction ("Inference
 * optimization", Step 3 prefix cache and exercise 4; "Continuous batching and
 * PagedAttention", section 3, shared read-only blocks).  An entry is one full
 * block_size-token block of a prompt, reached from the root by the prompt's blocks
 * before it; the cache holds one reference on each cached block.  A lookup matches at
 * most (num_tokens - 1) / block_size blocks (the last prompt token is always
 * computed).  Entries carry last-use stamps; only leaves are evicted, least recently
 * used first; an insertion evicts down to max_entries.  Host memory only.
 * ------------------------------------------------------------------------------------ */
typedef struct pkv_prefix_cache pkv_prefix_cache;
int pkv_pcache_create(pkv_pool *pool, int max_entries, pkv_prefix_cache **out);
/* Releases the cache's references; the pool must outlive the cache. */
void pkv_pcache_destroy(pkv_prefix_cache *cache);
/* Blocks of the longest cached prefix of tokens[num_tokens] into blocks[max_blocks];
 * returns how many (>= 0) or an error.  No side effect. */
int pkv_pcache_lookup(const pkv_prefix_cache *cache, const int32_t *tokens, int num_tokens,
                      int32_t *blocks, int max_blocks);
/* Record that a request uses the first num_matched matched blocks: touches them and
 * counts the lookup in the statistics. */
int pkv_pcache_use(pkv_prefix_cache *cache, const int32_t *tokens, int num_tokens,
                   int num_matched);
/* Cache the full blocks of a computed prompt (table: its block table, at least
 * num_tokens / block_size entries, all allocated), touching each, then evict down to
 * max_entries. */
int pkv_pcache_insert(pkv_prefix_cache *cache, const int32_t *tokens, int num_tokens,
                      const int32_t *table, int table_len);
/* Evict the least recently used leaf whose block only the cache holds: 1 if one was
 * evicted (one pool block freed), 0 if none. */
int pkv_pcache_evict_free_one(pkv_prefix_cache *cache);
/* out[6] = lookups, lookups with a hit, tokens looked up, tokens matched, entries,
 * evictions. */
int pkv_pcache_stats(const pkv_prefix_cache *cache, int64_t *out);

/* ------------------------------------------------------------------------------------
 * Continuous-batching scheduler with chunked prefill ("Continuous batching and
 * PagedAttention", section 2: iteration-level scheduling, chunked prefill with a
 * per-step token budget; "Inference optimization", continuous batching and exercise 2).
 * Each step: (1) retire requests that produced all their output tokens (free their
 * blocks); (2) one decode token for every running request whose prompt is complete,
 * in admission order; (3) the next prefill chunk of requests still prefilling, while
 * the step's token budget lasts; (4) admit waiting requests first come first served
 * while fewer than max_num_seqs run and budget is left (static_batching != 0: only into
 * an empty batch).  Admission starts a request's table with its prefix-cache match.
 * Out of blocks: evict an unused cached block, else preempt the most recently admitted
 * request (its blocks are freed; it is recomputed from the start when readmitted).
 * A request's KV holds its prompt and all output tokens but the last; the step that
 * completes a prompt samples the first output token and caches the prompt's full
 * blocks.  Sequence ids in the pool are the request ids.
 * ------------------------------------------------------------------------------------ */
typedef struct pkv_sched pkv_sched;

/* One step's work, in host memory owned by the scheduler (valid until the next step).
 * Entries: decode entries (query_len 1) first, then prefill chunks. */
typedef struct {
  int num_seqs;                 /* scheduled sequences                              */
  int num_decode;               /* of which decode entries (the first num_decode)   */
  int num_tokens;               /* new tokens = sum of query_lens                   */
  int max_blocks;               /* row length of block_tables                       */
  int num_cow;                  /* copy-on-write pairs to apply before the writes   */
  int finished;                 /* requests retired at the start of this step       */
  int preempted;                /* requests preempted during this step              */
  int running;                  /* running requests after the step                  */
  int waiting;                  /* waiting requests after the step                  */
  const int64_t *seq_ids;       /* [num_seqs]                                       */
  const int32_t *query_lens;    /* [num_seqs] new tokens per sequence               */
  const int32_t *context_lens;  /* [num_seqs] tokens after the step's writes        */
  const int32_t *query_start;   /* [num_seqs + 1] offsets of each sequence's tokens */
  const int64_t *slot_mapping;  /* [num_tokens] slots of the new tokens, in order   */
  const int32_t *block_tables;  /* [num_seqs][max_blocks], unused entries -1        */
  const int32_t *cow_pairs;     /* [num_cow][2] (src, dst)                          */
} pkv_step_plan;

typedef struct {
  int64_t steps, finished, preemptions, decode_tokens, prefill_tokens, busy_steps;
  double fill_sum;              /* sum over steps of running / max_num_seqs         */
  double busy_fill_sum;         /* the same over steps that end with requests waiting */
  int64_t slots_held;           /* sum over steps and running requests of token slots */
  int64_t slots_unused;         /* ... of which not holding a token (internal waste)  */
} pkv_sched_stats;

/* cache may be NULL (no prefix caching); it must use the same pool.
 * max_batched_tokens >= max_num_seqs. */
int pkv_sched_create(pkv_pool *pool, pkv_prefix_cache *cache, int max_num_seqs,
                     int max_batched_tokens, int static_batching, pkv_sched **out);
/* Frees the blocks of requests still running. */
void pkv_sched_destroy(pkv_sched *sched);
/* Queue a request (prompt_tokens may be NULL: the request then bypasses the cache). */
int pkv_sched_add_request(pkv_sched *sched, int64_t id, int prompt_len,
                          const int32_t *prompt_tokens, int output_len);
/* Run one step; fills *plan.  Returns the number of scheduled sequences (0 when
 * nothing is left to do), or PKV_ERR_OOM when requests remain but none can progress
 * (the pool is too small for the request at the head of the queue). */
int pkv_sched_step(pkv_sched *sched, pkv_step_plan *plan);
/* The last step's plan packed for one host-to-device copy.  Every array sits at a fixed
 * 256-byte aligned offset that depends only on the capacities (max_tokens new tokens,
 * max_seqs sequences, block-table rows of table_stride entries, -1 past the sequence's
 * blocks), so device views of a staging buffer can be made once.  Besides the plan's
 * arrays it holds, per new token, the request id, the position and the prompt token at
 * that position (-1 past the prompt: a generated token, which the caller knows), and per
 * prefill chunk its offset and the row of its last token within the prefill rows. */
typedef struct {
  int64_t slot_mapping;    /* int64 [num_tokens]                                       */
  int64_t token_seq;       /* int64 [num_tokens] request id of each new token          */
  int64_t last_rows;       /* int64 [chunks] last row of each prefill chunk            */
  int64_t block_tables;    /* int32 [num_seqs][table_stride]                           */
  int64_t context_lens;    /* int32 [num_seqs]                                         */
  int64_t cow_pairs;       /* int32 [num_cow][2]                                       */
  int64_t prefill_start;   /* int32 [chunks + 1] chunk offsets within the prefill rows */
  int64_t token_ids;       /* int32 [num_tokens] prompt token, or -1                   */
  int64_t positions;       /* int32 [num_tokens]                                       */
  int64_t kv_rows;         /* int64 [num_tokens] left for pkv_step_synthetic_rows      */
  int64_t q_rows;          /* int64 [num_tokens] left for pkv_step_synthetic_rows      */
  int64_t total;           /* bytes the layout spans                                   */
  int num_seqs, num_decode, num_tokens, num_cow;
  int decode_max_context;  /* largest context among the decode entries                 */
  int prefill_max_query;   /* longest prefill chunk                                    */
  int outputs;             /* output tokens the step yields (decode entries + chunks
                              that complete their prompt)                              */
} pkv_step_pack;

/* Writes the last pkv_sched_step's plan into buf (host memory, e.g. pinned staging)
 * in the pkv_step_pack layout and fills *pack.  PKV_ERR_ARG if a count exceeds its
 * capacity or buf_bytes < pack->total (the offsets and pack->total are filled even
 * then); buf == NULL returns PKV_ERR_NULL after filling the layout. */
int pkv_sched_pack(const pkv_sched *sched, void *buf, int64_t buf_bytes, int max_tokens,
                   int max_seqs, int table_stride, pkv_step_pack *pack);
/* The synthetic model of the serving benchmark and tests (it stands in for the layers
 * that would produce each new token's q/K/V on the device): over a packed step in buf,
 * every token id of -1 becomes the seeded generated id (rid * 7777 + pos * 131) mod
 * 32000, and each new token gets the rows of its K/V in a table of table_rows rows,
 * (token * 1000003 + pos * 7919) mod table_rows, and of its query,
 * (rid * 2654435761 + pos * 40503) mod table_rows.  Not part of the method. */
int pkv_step_synthetic_rows(void *buf, const pkv_step_pack *pack, int64_t table_rows);

/*
 * paged_gather_rows -- dst row i = src row idx[i] for i < n, rows of row_bytes bytes (a
 * multiple of 16; dst and src 16-byte aligned, device memory; idx int64 [n], device).
 * An index outside [0, src_rows) sets PKV_DEV_BAD_ROW and leaves that destination row
 * unwritten.  n == 0 does nothing.  PKV_ERR_SHAPE when n * row_bytes / 16 >= 2^31.
 * The serving step uses it to pick each chunk's last prefill row and the synthetic
 * model's q/K/V rows.
 */
int paged_gather_rows(void *dst, const void *src, const int64_t *idx, int n, int64_t src_rows,
                      int row_bytes, int32_t *err_flag, void *stream);

/*
 * pkv_step_launch -- the device half of one packed serving step, queued on `stream` by
 * one call (the loop of "Continuous batching and PagedAttention", section 2: every step
 * runs the decode entries and the prefill chunks the scheduler picked):
 *   1. one copy of the packed step (pack->total bytes, pkv_sched_pack) from
 *      io->host_stage[slot] to io->dev_stage;
 *   2. if io->k_table != NULL (the synthetic model): one launch gathering, per new token
 *      t, k_new[t] = k_table[kv_rows[t]], v_new[t] = v_table[kv_rows[t]] and
 *      q[t] = q_table[q_rows[t]] (pkv_step_synthetic_rows); with k_table NULL the
 *      caller has filled k_new, v_new and q (rows in the pack's token order);
 *   3. paged_decode_step: the step's copy-on-write pairs, the paged write of every new
 *      token, decode attention of the num_decode decode entries into out rows
 *      0 .. num_decode - 1;
 *   4. with prefill chunks: paged_attention_prefill of the chunk rows (new tokens
 *      num_decode .. num_tokens - 1) into prefill_out, then the last row of chunk c
 *      gathered into out row num_decode + c;
 *   5. one copy of out rows 0 .. num_seqs - 1 to io->out_host[slot].
 * events: NULL, or three cudaEvent_t (each may be NULL) recorded on the stream before
 * step 1, before step 3 and after step 3.  All buffers are the caller's and stay
 * untouched by the host; host_stage[slot] and out_host[slot] must be pinned and must
 * not be reused before the stream has passed this step.  A pack with more tokens or
 * sequences than io's capacities, or a total above stage_bytes, returns PKV_ERR_SHAPE
 * and queues nothing; otherwise the first failing call's code is returned and nothing
 * after it is queued.  Device-side errors are ORed into io->err_flag as by the calls.
 */
typedef struct {
  void *host_stage[2];        /* pinned staging buffers, one per in-flight step        */
  void *dev_stage;            /* device copy of a staging buffer (stage_bytes)         */
  int64_t stage_bytes;
  const uint16_t *k_table;    /* bf16 [table_rows][num_kv_heads][head_dim], or NULL    */
  const uint16_t *v_table;    /* bf16 [table_rows][num_kv_heads][head_dim]             */
  const uint16_t *q_table;    /* bf16 [table_rows][num_q_heads][head_dim]              */
  int64_t table_rows;
  uint16_t *k_new, *v_new;    /* bf16 [max_tokens][num_kv_heads][head_dim]             */
  uint16_t *q;                /* bf16 [max_tokens][num_q_heads][head_dim]              */
  uint16_t *prefill_out;      /* bf16 [max_tokens][num_q_heads][head_dim]              */
  uint16_t *out;              /* bf16 [max_seqs][num_q_heads][head_dim], device        */
  uint16_t *out_host[2];      /* the same shape, pinned host, one per in-flight step   */
  uint16_t *k_cache, *v_cache;/* bf16 [num_blocks][num_kv_heads][16][head_dim]         */
  int max_tokens, max_seqs;   /* capacities (the pkv_sched_pack capacities)            */
  int num_blocks, num_q_heads, num_kv_heads, head_dim, block_size;
  int table_stride;           /* entries per block-table row in the pack               */
  int partition_size;
  float scale;
  void *workspace;            /* decode workspace for max_seqs sequences               */
  size_t workspace_bytes;
  int32_t *err_flag;          /* device word (may be NULL)                             */
} pkv_step_io;
int pkv_step_launch(const pkv_step_io *io, const pkv_step_pack *pack, int slot,
                    void *const *events, void *stream);

/*
 * pkv_engine_step -- one whole iteration of the serving loop from the host: pkv_sched_step
 * on `sched`, pkv_sched_pack of its plan into io->host_stage[slot] (capacities
 * io->max_tokens, io->max_seqs, io->table_stride, io->stage_bytes), then, if
 * io->k_table != NULL, pkv_step_synthetic_rows over it (io->table_rows), then
 * pkv_step_launch(io, pack, slot, events, stream).  Fills *pack.  Returns the number of
 * scheduled sequences (pkv_sched_step's value; the step launches nothing when
 * pack->num_tokens == 0, and no event is then recorded), or the first failing call's
 * code.  host_stage[slot] must not be in use by an earlier step still on the stream.
 */
int pkv_engine_step(pkv_sched *sched, const pkv_step_io *io, pkv_step_pack *pack, int slot,
                    void *const *events, void *stream);
int pkv_sched_done(const pkv_sched *sched);  /* 1 when no request is waiting or running */
int pkv_sched_get_stats(const pkv_sched *sched, pkv_sched_stats *out);

/*
 * pkv_selftest_bounded_wait -- exercises the kernels' failure path without a fault.
 * Every wait inside the library's kernels is bounded (about one second); when one gives
 * up, the kernel ORs PKV_DEV_TIMEOUT into the caller's error word and returns, and the
 * context stays usable.  This call launches one thread that waits, with the same wait
 * helpers (use_spin != 0: the polling variant) and a limit of limit_cycles clock cycles
 * (0 < limit_cycles <= about one second), on an mbarrier phase that nothing completes.
 * err_flag: int32 device word, ORed with PKV_DEV_TIMEOUT when the wait gives up.
 * result: int64 device array of 3: [0] 1 if the wait succeeded (never), [1] cycles
 * spent, [2] the CTA abort flag after the wait.  Returns PKV_ERR_NULL for a null pointer,
 * PKV_ERR_SHAPE for a limit out of range, PKV_ERR_CUDA if the launch failed, else PKV_OK.
 */
int pkv_selftest_bounded_wait(int32_t *err_flag, long long *result, long long limit_cycles,
                              int use_spin, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
