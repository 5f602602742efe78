/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the paged KV-cache decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark may load this library.  It shares no code, header, table or
 * helper with the CUDA library; it reads the same input bytes and nothing else.
 *
 * What it computes, and where the pages state it:
 *
 *  - oracle_kv_write: the new token's K/V is computed once and appended to the cache
 *    ("Inference optimization", section "KV cache": only the N-th token's K/V is
 *    computed and concatenated with tokens 1..N-1; section "Step 1: KV cache", the
 *    KVCache.update method).  With a paged cache the append lands in the physical
 *    block the block table names ("Continuous batching and PagedAttention", section 3
 *    PagedAttention: per-request block table, logical block -> physical block).
 *    Slot = physical_block * block_size + offset.  A negative slot is skipped.
 *
 *  - oracle_block_copy: copy-on-write makes a private copy of a shared block when a
 *    request diverges ("Continuous batching and PagedAttention", section 3, the
 *    copy-on-write sharing paragraph).  Byte copy of every KV head of the block.
 *
 *  - oracle_attention: Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V
 *    ("System-level optimization: batching, PagedAttention and FlashAttention",
 *    section 3.1, the attention equation; section 3.3 passes scale = head_dim**-0.5).
 *    Each sequence's blocks are first gathered into a contiguous K/V (the contiguous
 *    KVCache view of "Inference optimization", Step 1), then the textbook softmax
 *    is taken in fp64 with the maximum subtracted.  No partitioning, no tiling.
 *    Query head h reads KV head h / (Hq/Hkv) (grouped-query attention: 64 query
 *    heads share 8 KV heads, "Inference optimization", exercise 3).
 *
 *  - oracle_attention_prefill: the same softmax for several new tokens per sequence
 *    (chunked prefill), each seeing the tokens up to its own position (causal); see
 *    the comment above the function.
 *
 * Layouts (all row-major, element type bf16 stored as uint16 bit patterns):
 *   q[S][Hq][D], k_cache/v_cache[NB][Hkv][block_size][D],
 *   block_tables[S][MB] int32, context_lens[S] int32, out[S][Hq][D] fp64.
 *
 * Return codes: 0 ok, -1 bad sizes, -2 index out of range (nothing is read or written
 * outside the buffers; the whole call is abandoned at the first bad index).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> fp64 is exact: the bf16 bits are the top half of an fp32. */
static double bf16_to_f64(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_abi_version(void) { return 2; }  /* 2: E4M3 scales per KV head */

int oracle_kv_write(uint16_t *k_cache, uint16_t *v_cache,
                    const uint16_t *k_new, const uint16_t *v_new,
                    const int64_t *slot_mapping, int num_tokens,
                    int num_blocks, int num_kv_heads, int head_dim, int block_size) {
    if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
        return -1;
    const int64_t num_slots = (int64_t)num_blocks * block_size;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) return -2;
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            size_t dst = (((size_t)block * num_kv_heads + h) * block_size + offset) * head_dim;
            size_t src = ((size_t)t * num_kv_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d) {
                k_cache[dst + d] = k_new[src + d];
                v_cache[dst + d] = v_new[src + d];
            }
        }
    }
    return 0;
}

int oracle_block_copy(uint16_t *k_cache, uint16_t *v_cache, const int32_t *pairs, int num_pairs,
                      int num_blocks, int num_kv_heads, int head_dim, int block_size) {
    if (num_pairs < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
        return -1;
    const size_t block_elems = (size_t)num_kv_heads * block_size * head_dim;
    for (int i = 0; i < num_pairs; ++i) {
        int32_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return -2;
        for (size_t e = 0; e < block_elems; ++e) {
            k_cache[(size_t)dst * block_elems + e] = k_cache[(size_t)src * block_elems + e];
            v_cache[(size_t)dst * block_elems + e] = v_cache[(size_t)src * block_elems + e];
        }
    }
    return 0;
}

/* One (sequence, query head) output.  kc/vc are caller scratch of ctx*head_dim doubles. */
static int attend_one(double *out, const uint16_t *q, const uint16_t *k_cache,
                      const uint16_t *v_cache, const int32_t *block_table, int ctx,
                      int max_blocks, int head, int num_q_heads, int num_kv_heads, int head_dim,
                      int block_size, int num_blocks, double scale,
                      double *kc, double *vc, double *x) {
    const int group = num_q_heads / num_kv_heads;
    const int kv_head = head / group;
    if (ctx > max_blocks * block_size) return -2;
    /* Gather the logical token sequence into a contiguous K/V. */
    for (int t = 0; t < ctx; ++t) {
        int32_t block = block_table[t / block_size];
        if (block < 0 || block >= num_blocks) return -2;
        int offset = t % block_size;
        size_t row = (((size_t)block * num_kv_heads + kv_head) * block_size + offset) * head_dim;
        for (int d = 0; d < head_dim; ++d) {
            kc[(size_t)t * head_dim + d] = bf16_to_f64(k_cache[row + d]);
            vc[(size_t)t * head_dim + d] = bf16_to_f64(v_cache[row + d]);
        }
    }
    if (ctx == 0) {
        for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
        return 0;
    }
    /* Scores x_t = scale * q . k_t */
    double m = -INFINITY;
    for (int t = 0; t < ctx; ++t) {
        double acc = 0.0;
        for (int d = 0; d < head_dim; ++d) acc += bf16_to_f64(q[d]) * kc[(size_t)t * head_dim + d];
        x[t] = scale * acc;
        if (x[t] > m) m = x[t];
    }
    /* Softmax weights and the weighted sum of V. */
    double denom = 0.0;
    for (int t = 0; t < ctx; ++t) {
        x[t] = exp(x[t] - m);
        denom += x[t];
    }
    /* o[d] = sum_t w_t V[t][d] / sum_t w_t: for every d the terms are added in
     * increasing t; t is the outer loop so that V is read one row at a time. */
    for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
    for (int t = 0; t < ctx; ++t) {
        const double *vt = vc + (size_t)t * head_dim;
        for (int d = 0; d < head_dim; ++d) out[d] += x[t] * vt[d];
    }
    for (int d = 0; d < head_dim; ++d) out[d] /= denom;
    return 0;
}

/*
 * out[S][Hq][D] in fp64.  If `sel` is non-NULL only the `nsel` (sequence, head) pairs
 * sel[2i], sel[2i+1] are computed, and out is then [nsel][D].  nthreads <= 0 means
 * one thread.  Returns 0, -1 (bad sizes) or -2 (index out of range).
 */
int oracle_attention(double *out, const uint16_t *q, const uint16_t *k_cache,
                     const uint16_t *v_cache, const int32_t *block_tables,
                     const int32_t *context_lens, int num_seqs, int max_blocks,
                     int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                     int num_blocks, double scale, const int32_t *sel, int nsel, int nthreads) {
    if (num_seqs < 0 || max_blocks <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || block_size <= 0 || num_blocks <= 0 || num_q_heads % num_kv_heads != 0)
        return -1;
    const int npairs = sel ? nsel : num_seqs * num_q_heads;
    int max_ctx = 0;
    for (int s = 0; s < num_seqs; ++s) {
        if (context_lens[s] < 0) return -1;
        if (context_lens[s] > max_ctx) max_ctx = context_lens[s];
    }
    if (nthreads <= 0) nthreads = 1;
    int status = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(nthreads)
#endif
    {
        size_t n = (size_t)(max_ctx > 0 ? max_ctx : 1);
        double *kc = (double *)malloc(n * head_dim * sizeof(double));
        double *vc = (double *)malloc(n * head_dim * sizeof(double));
        double *x = (double *)malloc(n * sizeof(double));
        int local = (kc && vc && x) ? 0 : -3;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int i = 0; i < npairs; ++i) {
            if (local) continue;
            int s = sel ? sel[2 * i] : i / num_q_heads;
            int h = sel ? sel[2 * i + 1] : i % num_q_heads;
            if (s < 0 || s >= num_seqs || h < 0 || h >= num_q_heads) { local = -2; continue; }
            int rc = attend_one(out + (size_t)i * head_dim,
                                q + ((size_t)s * num_q_heads + h) * head_dim, k_cache, v_cache,
                                block_tables + (size_t)s * max_blocks, context_lens[s], max_blocks,
                                h, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                scale, kc, vc, x);
            if (rc) local = rc;
        }
#ifdef _OPENMP
#pragma omp critical
#endif
        if (local && !status) status = local;
        free(kc);
        free(vc);
        free(x);
    }
    return status;
}

/* KV bytes one token occupies: 2 (K and V) x layers x KV heads x head_dim x bytes per
 * element ("Inference optimization", section "KV cache", the memory formula). */
int64_t oracle_kv_bytes_per_token(int layers, int kv_heads, int head_dim, int bytes_per_elem) {
    return (int64_t)2 * layers * kv_heads * head_dim * bytes_per_elem;
}

/* ------------------------------------------------------------------------------------
 * FP8 (E4M3) KV cache.  "Continuous batching and PagedAttention", section 4 (vLLM's
 * kv_cache_dtype="fp8" option) and "Inference optimization", exercise 1 (quantised KV
 * caches hold more concurrent requests).  The pages name the format only; the codec
 * below follows the OCP 8-bit floating point E4M3 definition: 1 sign bit, 4 exponent
 * bits (bias 7), 3 mantissa bits, no infinities, S.1111.111 is NaN, largest finite
 * value 448.  Rounding is to nearest, ties to even; a finite value beyond 448 saturates
 * to +-448 (the "satfinite" convention).  A cache element holds
 * code = E4M3(bf16_value / scale), the division taken in fp32, and stands for
 * decode(code) * scale.  A scale belongs to one KV head of one cache (k_scales[h],
 * v_scales[h]): the per-tensor scheme is the case of equal entries.  The pages leave
 * the scale's granularity open; per-KV-head scales follow each head's own range.
 * Layouts: K codes [NB][Hkv][block_size][D] like the bf16 cache; V codes transposed
 * within each block, [NB][Hkv][D][block_size] (an interface choice of the E4M3 cache).
 * ------------------------------------------------------------------------------------ */
double oracle_e4m3_decode(uint8_t c) {
    const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double v = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

uint8_t oracle_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);            /* a = f * 2^e2, f in [0.5, 1): a = 1.xxx * 2^(e2 - 1) */
    int E = e2 - 1;
    if (E < -6) E = -6;       /* subnormal range shares the spacing of 2^-6 */
    const double spacing = ldexp(1.0, E - 3);
    const double r = rint(a / spacing); /* default rounding mode: nearest, ties to even */
    const double v = r * spacing;
    if (v >= 448.0) return sign | 0x7E;
    if (v == 0.0) return sign;
    if (v < ldexp(1.0, -6)) return sign | (uint8_t)(v / ldexp(1.0, -9));
    int ev;
    frexp(v, &ev);
    const int Ev = ev - 1;
    const int mant = (int)((v / ldexp(1.0, Ev) - 1.0) * 8.0);
    return sign | (uint8_t)(((Ev + 7) << 3) | mant);
}

int oracle_kv_write_fp8(uint8_t *k_cache, uint8_t *v_cache, const uint16_t *k_new,
                        const uint16_t *v_new, const int64_t *slot_mapping, int num_tokens,
                        int num_blocks, int num_kv_heads, int head_dim, int block_size,
                        const float *k_scales, const float *v_scales) {
    if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        !k_scales || !v_scales)
        return -1;
    const int64_t num_slots = (int64_t)num_blocks * block_size;
    for (int t = 0; t < num_tokens; ++t)
        if (slot_mapping[t] >= num_slots) return -2;
    /* tokens are independent (distinct slots), so the loop may run on several threads */
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        int64_t block = slot / block_size, offset = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            size_t dst = (((size_t)block * num_kv_heads + h) * block_size + offset) * head_dim;
            size_t vbase = ((size_t)block * num_kv_heads + h) * head_dim * block_size + offset;
            size_t src = ((size_t)t * num_kv_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d) {
                float kx = (float)bf16_to_f64(k_new[src + d]);
                float vx = (float)bf16_to_f64(v_new[src + d]);
                k_cache[dst + d] = oracle_e4m3_encode(kx / k_scales[h]);
                v_cache[vbase + (size_t)d * block_size] = oracle_e4m3_encode(vx / v_scales[h]);
            }
        }
    }
    return 0;
}

int oracle_block_copy_fp8(uint8_t *k_cache, uint8_t *v_cache, const int32_t *pairs, int num_pairs,
                          int num_blocks, int num_kv_heads, int head_dim, int block_size) {
    if (num_pairs < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
        return -1;
    const size_t block_elems = (size_t)num_kv_heads * block_size * head_dim;
    for (int i = 0; i < num_pairs; ++i) {
        int32_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return -2;
        memcpy(k_cache + (size_t)dst * block_elems, k_cache + (size_t)src * block_elems, block_elems);
        memcpy(v_cache + (size_t)dst * block_elems, v_cache + (size_t)src * block_elems, block_elems);
    }
    return 0;
}

/* Decode attention over an E4M3 cache: every element of KV head g is
 * decode(code) * k_scales[g] (K) or decode(code) * v_scales[g] (V) in fp64; the rest is
 * the same textbook softmax as oracle_attention. */
int oracle_attention_fp8(double *out, const uint16_t *q, const uint8_t *k_cache,
                         const uint8_t *v_cache, const int32_t *block_tables,
                         const int32_t *context_lens, int num_seqs, int max_blocks,
                         int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, double scale, const double *k_scales,
                         const double *v_scales, const int32_t *sel, int nsel, int nthreads) {
    if (num_seqs < 0 || max_blocks <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || block_size <= 0 || num_blocks <= 0 || num_q_heads % num_kv_heads != 0 ||
        !k_scales || !v_scales)
        return -1;
    const int npairs = sel ? nsel : num_seqs * num_q_heads;
    const int group = num_q_heads / num_kv_heads;
    int max_ctx = 0;
    for (int s = 0; s < num_seqs; ++s) {
        if (context_lens[s] < 0) return -1;
        if (context_lens[s] > max_ctx) max_ctx = context_lens[s];
    }
    if (nthreads <= 0) nthreads = 1;
    int status = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(nthreads)
#endif
    {
        size_t n = (size_t)(max_ctx > 0 ? max_ctx : 1);
        double *kc = (double *)malloc(n * head_dim * sizeof(double));
        double *vc = (double *)malloc(n * head_dim * sizeof(double));
        double *x = (double *)malloc(n * sizeof(double));
        int local = (kc && vc && x) ? 0 : -3;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int i = 0; i < npairs; ++i) {
            if (local) continue;
            int s = sel ? sel[2 * i] : i / num_q_heads;
            int h = sel ? sel[2 * i + 1] : i % num_q_heads;
            if (s < 0 || s >= num_seqs || h < 0 || h >= num_q_heads) { local = -2; continue; }
            const int ctx = context_lens[s], kv_head = h / group;
            const int32_t *table = block_tables + (size_t)s * max_blocks;
            double *o = out + (size_t)i * head_dim;
            const uint16_t *qh = q + ((size_t)s * num_q_heads + h) * head_dim;
            const double k_scale = k_scales[kv_head], v_scale = v_scales[kv_head];
            if (ctx > max_blocks * block_size) { local = -2; continue; }
            int bad = 0;
            for (int t = 0; t < ctx && !bad; ++t) {
                int32_t block = table[t / block_size];
                if (block < 0 || block >= num_blocks) { bad = 1; break; }
                size_t row = (((size_t)block * num_kv_heads + kv_head) * block_size +
                              t % block_size) * head_dim;
                size_t vcol = ((size_t)block * num_kv_heads + kv_head) * head_dim * block_size +
                              t % block_size;
                for (int d = 0; d < head_dim; ++d) {
                    kc[(size_t)t * head_dim + d] = oracle_e4m3_decode(k_cache[row + d]) * k_scale;
                    vc[(size_t)t * head_dim + d] =
                        oracle_e4m3_decode(v_cache[vcol + (size_t)d * block_size]) * v_scale;
                }
            }
            if (bad) { local = -2; continue; }
            if (ctx == 0) {
                for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
                continue;
            }
            double m = -INFINITY;
            for (int t = 0; t < ctx; ++t) {
                double acc = 0.0;
                for (int d = 0; d < head_dim; ++d) acc += bf16_to_f64(qh[d]) * kc[(size_t)t * head_dim + d];
                x[t] = scale * acc;
                if (x[t] > m) m = x[t];
            }
            double denom = 0.0;
            for (int t = 0; t < ctx; ++t) {
                x[t] = exp(x[t] - m);
                denom += x[t];
            }
            /* as in attend_one: per d, terms added in increasing t, V read by rows */
            for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
            for (int t = 0; t < ctx; ++t) {
                const double *vt = vc + (size_t)t * head_dim;
                for (int d = 0; d < head_dim; ++d) o[d] += x[t] * vt[d];
            }
            for (int d = 0; d < head_dim; ++d) o[d] /= denom;
        }
#ifdef _OPENMP
#pragma omp critical
#endif
        if (local && !status) status = local;
        free(kc);
        free(vc);
        free(x);
    }
    return status;
}

/* ------------------------------------------------------------------------------------
 * Chunked prefill: several new query tokens per sequence.  "Continuous batching and
 * PagedAttention", section 2 (continuous batching): a long prefill inserted into a
 * decode batch stalls every decoding request, and the first remedy is to cut the
 * prefill into chunks spread over several iterations.  A chunk's tokens attend
 * causally ("System-level optimization", section 3.3 calls the library routine with
 * is_causal=True): a query token at position p sees the cached tokens 0..p, itself
 * included, and nothing after it.
 *
 * Sequence s contributes L = query_start[s+1] - query_start[s] query tokens, rows
 * query_start[s] .. query_start[s+1]-1 of q and out ([num_tokens][Hq][D]); they are
 * the last L of its context_lens[s] tokens, already in the cache, so query token i
 * (0 <= i < L) sits at position p = context_lens[s] - L + i.  Each (token, head) row is
 * the textbook softmax over the first p + 1 tokens, exactly as oracle_attention computes
 * a decode row with context p + 1.  sel, if given, lists nsel (token, head) pairs and
 * out is then [nsel][D].
 * ------------------------------------------------------------------------------------ */
int oracle_attention_prefill(double *out, const uint16_t *q, const uint16_t *k_cache,
                             const uint16_t *v_cache, const int32_t *block_tables,
                             const int32_t *context_lens, const int32_t *query_start,
                             int num_seqs, int num_tokens, int max_blocks, int num_q_heads,
                             int num_kv_heads, int head_dim, int block_size, int num_blocks,
                             double scale, const int32_t *sel, int nsel, int nthreads) {
    if (num_seqs < 0 || num_tokens < 0 || max_blocks <= 0 || num_q_heads <= 0 ||
        num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0 ||
        num_q_heads % num_kv_heads != 0)
        return -1;
    if (query_start[0] != 0 || query_start[num_seqs] != num_tokens) return -1;
    int max_ctx = 0;
    for (int s = 0; s < num_seqs; ++s) {
        const int L = query_start[s + 1] - query_start[s];
        if (L < 0 || context_lens[s] < L) return -1;
        if (context_lens[s] > max_ctx) max_ctx = context_lens[s];
    }
    const int npairs = sel ? nsel : num_tokens * num_q_heads;
    if (nthreads <= 0) nthreads = 1;
    int status = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(nthreads)
#endif
    {
        size_t n = (size_t)(max_ctx > 0 ? max_ctx : 1);
        double *kc = (double *)malloc(n * head_dim * sizeof(double));
        double *vc = (double *)malloc(n * head_dim * sizeof(double));
        double *x = (double *)malloc(n * sizeof(double));
        int local = (kc && vc && x) ? 0 : -3;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int i = 0; i < npairs; ++i) {
            if (local) continue;
            const int tok = sel ? sel[2 * i] : i / num_q_heads;
            const int h = sel ? sel[2 * i + 1] : i % num_q_heads;
            if (tok < 0 || tok >= num_tokens || h < 0 || h >= num_q_heads) { local = -2; continue; }
            int s = 0; /* the sequence whose rows hold token tok */
            while (query_start[s + 1] <= tok) ++s;
            const int L = query_start[s + 1] - query_start[s];
            const int pos = context_lens[s] - L + (tok - query_start[s]);
            int rc = attend_one(out + (size_t)i * head_dim,
                                q + ((size_t)tok * num_q_heads + h) * head_dim, k_cache, v_cache,
                                block_tables + (size_t)s * max_blocks, pos + 1, max_blocks, h,
                                num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                scale, kc, vc, x);
            if (rc) local = rc;
        }
#ifdef _OPENMP
#pragma omp critical
#endif
        if (local && !status) status = local;
        free(kc);
        free(vc);
        free(x);
    }
    return status;
}
