// The device half of one continuous-batching step, queued by one host call, and the row
// gather it uses.
//
// The scheduler's plan for the step arrives packed (pkv_sched_pack) in pinned staging;
// pkv_step_launch copies it to the device in one copy and queues, on one stream, the
// new tokens' q/K/V rows, the fused decode step (copy-on-write, paged write, decode
// attention), the chunked prefill, the gather of each chunk's last row and one copy of
// what a sampler reads back to pinned memory.  Everything between the scheduler and the
// sampler is thus one call from the host, with no per-step allocation.
// Sources: "Continuous batching and PagedAttention", section 2 (iteration-level
// scheduling, chunked prefill) and section 3 (block tables, copy-on-write).
#include "pkv_common.cuh"

namespace pkv {
namespace {

int grid_for_rows(int64_t total, int threads) {
  const int64_t want = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)device_sm_count() * 8;  // grid-stride beyond this
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

// One gather: dst row i (row_vecs 16-byte vectors) <- src row idx[i], i < total / row_vecs.
struct RowGather {
  const uint4 *src;
  uint4 *dst;
  const int64_t *idx;
  int64_t src_rows;
  uint32_t total;     // vectors to move (rows * row_vecs), < 2^31
  uint32_t row_vecs;
};

struct RowGathers {
  RowGather g[3];
};

// blockIdx.y selects the gather; thread index v enumerates (row, vector) with the vector
// fastest, so both the reads of a source row and the writes of its destination row are
// coalesced.
__global__ void __launch_bounds__(256) gather_rows_kernel(RowGathers jobs, int32_t *err) {
  pdl_trigger();
  pdl_wait();
  const RowGather j = blockIdx.y == 0 ? jobs.g[0] : (blockIdx.y == 1 ? jobs.g[1] : jobs.g[2]);
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t v = blockIdx.x * blockDim.x + threadIdx.x; v < j.total; v += stride) {
    const uint32_t i = v / j.row_vecs, e = v - i * j.row_vecs;
    const int64_t r = j.idx[i];
    if (r < 0 || r >= j.src_rows) {
      if (e == 0) flag_error(err, PKV_DEV_BAD_ROW);
      continue;
    }
    j.dst[v] = ld_stream_v4(j.src + r * j.row_vecs + e);
  }
}

// Host-side checks and the launch of up to three gathers (n[k] rows each).
int launch_gathers(const RowGather *g, int count, int32_t *err, cudaStream_t st) {
  RowGathers jobs = {};
  uint32_t most = 0;
  int used = 0;
  for (int k = 0; k < count; ++k) {
    if (g[k].total == 0) continue;
    jobs.g[used++] = g[k];
    most = g[k].total > most ? g[k].total : most;
  }
  if (used == 0) return PKV_OK;
  const int threads = 256;
  const cudaError_t e = launch_pdl(gather_rows_kernel, dim3(grid_for_rows(most, threads), used),
                                   dim3(threads), 0, st, jobs, err);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// One gather's description from the C arguments; PKV_OK or the error to return.
int make_gather(void *dst, const void *src, const int64_t *idx, int n, int64_t src_rows,
                int row_bytes, RowGather *g) {
  if (n < 0 || row_bytes <= 0 || row_bytes % 16 != 0 || src_rows <= 0) return PKV_ERR_SHAPE;
  if ((int64_t)n * (row_bytes / 16) >= (int64_t)1 << 31) return PKV_ERR_SHAPE;
  *g = RowGather{};
  if (n == 0) return PKV_OK;
  if (!dst || !src || !idx) return PKV_ERR_NULL;
  if (!aligned16(dst) || !aligned16(src)) return PKV_ERR_ALIGN;
  *g = RowGather{static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), idx, src_rows,
                 (uint32_t)((int64_t)n * (row_bytes / 16)), (uint32_t)(row_bytes / 16)};
  return PKV_OK;
}

int record(void *const *events, int k, cudaStream_t st) {
  if (!events || !events[k]) return PKV_OK;
  return cudaEventRecord(static_cast<cudaEvent_t>(events[k]), st) == cudaSuccess ? PKV_OK
                                                                                   : PKV_ERR_CUDA;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

int paged_gather_rows(void *dst, const void *src, const int64_t *idx, int n, int64_t src_rows,
                      int row_bytes, int32_t *err_flag, void *stream) {
  RowGather g;
  const int rc = make_gather(dst, src, idx, n, src_rows, row_bytes, &g);
  if (rc != PKV_OK) return rc;
  return launch_gathers(&g, 1, err_flag, (cudaStream_t)stream);
}

int pkv_step_launch(const pkv_step_io *io, const pkv_step_pack *pk, int slot,
                    void *const *events, void *stream) {
  if (!io || !pk) return PKV_ERR_NULL;
  if (slot != 0 && slot != 1) return PKV_ERR_ARG;
  const int T = pk->num_tokens, S = pk->num_seqs, nd = pk->num_decode;
  if (T < 0 || S < 0 || nd < 0 || nd > S || T > io->max_tokens || S > io->max_seqs ||
      pk->total <= 0 || pk->total > io->stage_bytes)
    return PKV_ERR_SHAPE;
  if (T == 0) return PKV_OK;
  if (!io->host_stage[slot] || !io->dev_stage || !io->out || !io->out_host[slot] || !io->q ||
      !io->k_new || !io->v_new)
    return PKV_ERR_NULL;
  const cudaStream_t st = (cudaStream_t)stream;
  const int Hq = io->num_q_heads, Hkv = io->num_kv_heads, D = io->head_dim;
  const int q_row = Hq * D * 2, kv_row = Hkv * D * 2;  // bytes of one q / K row
  char *d = static_cast<char *>(io->dev_stage);
  int rc = record(events, 0, st);
  if (rc != PKV_OK) return rc;
  if (cudaMemcpyAsync(io->dev_stage, io->host_stage[slot], (size_t)pk->total,
                      cudaMemcpyHostToDevice, st) != cudaSuccess)
    return PKV_ERR_CUDA;
  // The synthetic model: the new tokens' q/K/V rows from its tables.
  if (io->k_table) {
    const int64_t *kvr = reinterpret_cast<const int64_t *>(d + pk->kv_rows);
    const int64_t *qr = reinterpret_cast<const int64_t *>(d + pk->q_rows);
    RowGather g[3];
    if ((rc = make_gather(io->k_new, io->k_table, kvr, T, io->table_rows, kv_row, &g[0])) ||
        (rc = make_gather(io->v_new, io->v_table, kvr, T, io->table_rows, kv_row, &g[1])) ||
        (rc = make_gather(io->q, io->q_table, qr, T, io->table_rows, q_row, &g[2])) ||
        (rc = launch_gathers(g, 3, io->err_flag, st)))
      return rc;
  }
  const int32_t *tables = reinterpret_cast<const int32_t *>(d + pk->block_tables);
  const int32_t *ctx = reinterpret_cast<const int32_t *>(d + pk->context_lens);
  if ((rc = record(events, 1, st))) return rc;
  rc = paged_decode_step(io->out, io->q, io->k_cache, io->v_cache, tables, ctx, nd,
                         io->table_stride, Hq, Hkv, D, io->block_size, io->num_blocks,
                         io->scale, io->partition_size, pk->decode_max_context, io->k_new,
                         io->v_new, reinterpret_cast<const int64_t *>(d + pk->slot_mapping), T,
                         pk->num_cow ? reinterpret_cast<const int32_t *>(d + pk->cow_pairs)
                                     : nullptr,
                         pk->num_cow, io->workspace, io->workspace_bytes, io->err_flag, stream);
  if (rc != PKV_OK) return rc;
  if ((rc = record(events, 2, st))) return rc;
  const int chunks = S - nd;
  if (chunks > 0) {
    const int rows = T - nd;  // prefill rows follow the decode rows
    if (!io->prefill_out) return PKV_ERR_NULL;
    rc = paged_attention_prefill(io->prefill_out, io->q + (size_t)nd * Hq * D, io->k_cache,
                                 io->v_cache, tables + (size_t)nd * io->table_stride, ctx + nd,
                                 reinterpret_cast<const int32_t *>(d + pk->prefill_start),
                                 chunks, rows, io->table_stride, Hq, Hkv, D, io->block_size,
                                 io->num_blocks, io->scale, pk->prefill_max_query, io->err_flag,
                                 stream);
    if (rc != PKV_OK) return rc;
    RowGather g;
    if ((rc = make_gather(io->out + (size_t)nd * Hq * D, io->prefill_out,
                          reinterpret_cast<const int64_t *>(d + pk->last_rows), chunks, rows,
                          q_row, &g)) ||
        (rc = launch_gathers(&g, 1, io->err_flag, st)))
      return rc;
  }
  if (cudaMemcpyAsync(io->out_host[slot], io->out, (size_t)S * q_row, cudaMemcpyDeviceToHost,
                      st) != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

int pkv_engine_step(pkv_sched *sched, const pkv_step_io *io, pkv_step_pack *pk, int slot,
                    void *const *events, void *stream) {
  if (!sched || !io || !pk) return PKV_ERR_NULL;
  if (slot != 0 && slot != 1) return PKV_ERR_ARG;
  pkv_step_plan plan;
  const int n = pkv_sched_step(sched, &plan);
  if (n < 0) return n;
  int rc = pkv_sched_pack(sched, io->host_stage[slot], io->stage_bytes, io->max_tokens,
                          io->max_seqs, io->table_stride, pk);
  if (rc != PKV_OK) return rc;
  if (pk->num_tokens == 0) return n;
  if (io->k_table && (rc = pkv_step_synthetic_rows(io->host_stage[slot], pk, io->table_rows)))
    return rc;
  rc = pkv_step_launch(io, pk, slot, events, stream);
  return rc != PKV_OK ? rc : n;
}

}  // extern "C"
