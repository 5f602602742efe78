// Internal interface between the decode-attention translation units.
#pragma once

#include "pkv_common.cuh"

namespace pkv {

constexpr int kChunk = 32;  // partitions one merge unit combines

// One work item is (sequence s, partition p) x (KV head g, query sub-group).  The plan
// kernel lists every non-empty partition as an int4 record {s, t0, t1, np} (tokens
// [t0, t1) of sequence s, which has np partitions), ordered by block count, largest
// first, so that round-robin dealing of records to CTAs balances load.  Partitions
// hold part_tokens tokens, or, when part_max > part_tokens, a power-of-two multiple of
// it chosen by the plan from the call's total context (written to *part_eff).
//
// The merge kernel works on units (sequence, group of 8 query heads, chunk of up to
// kChunk partitions), also listed by the plan; a sequence with several chunks leaves
// one result per chunk and head, and the warp that completes a head's last chunk (an
// arrival counter per sequence and head) merges those.
struct AttnArgs {
  uint16_t *out;                 // [S][Hq][D] bf16
  const uint16_t *q;             // [S][Hq][D] bf16
  const void *k_cache;           // [NB][Hkv][16][D] bf16 (or E4M3 codes when kv8)
  const void *v_cache;
  const int32_t *block_tables;   // [S][MB]
  const int32_t *context_lens;   // [S]
  int num_seqs, max_blocks, num_q_heads, num_kv_heads, group, num_blocks;
  int part_tokens;               // smallest partition size in tokens (multiple of 16)
  int part_max;                  // largest the plan may choose (part_tokens: exact size)
  int part_fine;                 // automatic size in steps of 1.5x / 1.33x (else 2x)
  int part_div;                  // automatic size: records per resident CTA aimed at
  int slots;                     // about the partition kernel's resident CTAs
  int max_parts;                 // partitions per sequence the workspace holds (of
                                 //   part_tokens tokens)
  int sub_groups;                // query sub-groups per KV head (group > kernel width)
  int max_chunks;                // ceil(max_parts / kChunk)
  float scale_log2;              // scale * log2(e) (* k_scale for an E4M3 cache)
  float v_scale;                 // multiplies every output (1 for a bf16 cache)
  int kv8;                       // the caches hold E4M3 codes instead of bf16
  const float *k_scales;         // [Hkv] per-KV-head E4M3 scales, or null (per cache:
  const float *v_scales;         //   scale_log2 and v_scale already hold them)
  // workspace
  int32_t *num_items;            // [1]
  int32_t *part_eff;             // [1] partition size the plan chose (read by the kernels)
  int32_t *work_next;            // [1] next record to claim (tensor-core kernel)
  int4 *items;                   // [S * max_parts] records {s, t0, t1, np}
  float *part_lse;               // [S][max_parts][Hq]   log2-sum-exp2 of the partition
  float *part_o;                 // [S][max_parts][Hq][D] normalised partial output
  int4 *units;                   // [S * head groups * max_chunks] {s, head group, chunk, np}
  int32_t *num_units;            // [1]
  int32_t *cnt_seq;              // [S][Hq] chunks merged per head (multi-chunk sequences)
  float *chunk_lse;              // [S][max_chunks][Hq]
  float *chunk_o;                // [S][max_chunks][Hq][D]
  int32_t *err;
};

// Workspace carving (256-byte aligned sections).
struct AttnWorkspace {
  size_t num_items_off, work_next_off, items_off, lse_off, o_off, units_off, num_units_off,
      cnt_seq_off, chunk_lse_off, chunk_o_off, total;
};
AttnWorkspace attn_workspace_layout(int num_seqs, int num_q_heads, int head_dim, int max_parts);

// Launchers (return a cudaError_t value).
int launch_attn_fma(const AttnArgs &a, int head_dim, int width, cudaStream_t st);
int launch_attn_mma(const AttnArgs &a, int head_dim, cudaStream_t st);

// One decode-attention call, validated and laid out over its workspace.
struct DecodeCall {
  AttnArgs a;
  int head_dim;
  bool use_mma;  // tensor-core partition kernel (else the CUDA-core one)
  int width;     // query rows per item of the CUDA-core kernel
  bool empty;    // nothing to launch (no sequences)
};

// Checks the arguments of a decode-attention call and fills *d.  Returns PKV_OK or the
// PKV_ERR_* code the entry points return; nothing is enqueued.
int decode_prepare(DecodeCall *d, uint16_t *out, const uint16_t *q, const void *k_cache,
                   const void *v_cache, const int32_t *block_tables, const int32_t *context_lens,
                   int num_seqs, int max_blocks_per_seq, int num_q_heads, int num_kv_heads,
                   int head_dim, int block_size, int num_blocks, float scale, int partition_size,
                   int max_context_len, void *workspace, size_t workspace_bytes,
                   int32_t *err_flag, bool kv8, float k_scale, float v_scale,
                   const float *k_scales, const float *v_scales);

// Enqueues the partition kernel and the merge of a prepared call; the call's plan
// (attn_plan_cta) must already be enqueued on `st`.  Returns PKV_OK or PKV_ERR_CUDA.
int decode_launch_after_plan(const DecodeCall &d, cudaStream_t st);

}  // namespace pkv
