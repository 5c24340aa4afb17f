/*
 * kf_oracle.c -- plain fp64 CPU oracle for split-KV paged decode attention.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file's library. It shares no code, header,
 * table or helper with the CUDA library; the only thing both sides share is
 * the seeded input generator.
 *
 * What it computes, and where each step comes from:
 *
 *  - Paged gather. Token t of request b lives in physical block
 *    block_tables[b][t / block_size], slot t % block_size; a block holds
 *    block_size x num_kv_heads x head_dim elements ("Disaggregated Inference
 *    Architecture: Paged KV-Cache Tiering, Chunked Prefill, and Asynchronous
 *    Overlap", ultrainstinct.tech, "Distributed Paged KV-Cache Tiering and
 *    Memory Layout" / "Physical Memory Block Layout"; the decode kernel
 *    "gathers over the physical blocks" through the block table, blog.lo0.es
 *    "The signature-dish specialist: vLLM's attention backend", "How the
 *    backend reads the paged KV").
 *
 *  - Decode attention of one query token over a token range: the plain
 *    definition softmax(q K^T * scale) V, in fp64, returned as a partial
 *    (o, lse) with o normalised and lse = m + ln(l). KernelFlume
 *    (academ.us/article/2606.29207), sections 3.1-3.2 and 5.1: an attention
 *    node computes local core attention over its token-range partition and
 *    returns partials (o_i, m_i, l_i). The pair (normalised o, lse) carries
 *    the same information, since l_i * e^{m_i} = e^{lse_i}.
 *
 *  - LSE merge of partials: ultrainstinct.tech page, "Mathematical
 *    Formulation of Chunked Attention", the updates m_new = max(m_prev, m_cur),
 *    l_new = e^{m_prev-m_new} l_prev + e^{m_cur-m_new} l_cur and the matching
 *    rescaled sum of O; KernelFlume section 5.1 states the merge equals
 *    attention over the full range.
 *
 *  - Append: the tail node writes the step's K_new/V_new at the request's
 *    next position before attending (KernelFlume section 3.2, "Local
 *    attention on the attention nodes").
 *
 *  - Multi-query (chunked prefill) attention: "Mathematical Formulation of
 *    Chunked Attention" on the ultrainstinct.tech page -- the query chunk k of a
 *    prompt attends to the keys of earlier chunks, held in the paged cache,
 *    without a mask, and to its own chunk's keys with causal masking. With
 *    the chunk already in the cache (L tokens in all, the chunk its last C),
 *    query j (0-based in the chunk) sits at position L - C + j and attends to
 *    tokens [0, L - C + j]. Non-causal: every query attends to all L tokens
 *    (the shared-prefix pass of cascade attention, "What FlashInfer brings:
 *    JIT and cascade attention" on blog.lo0.es: the prefix is attended once
 *    for all requests, then merged with each request's own suffix).
 *
 *  - FP8 KV cache: the decode posts on blog.lo0.es ("Quantised KV cache --
 *    --kv-cache-dtype fp8") store K/V in 8-bit floats with scales to halve the
 *    bytes decode reads. Here a cached element is an OCP FP8 E4M3 code c with
 *    a per-KV-head fp32 scale; its value is decode(c) * scale. The append
 *    quantises: c = E4M3 round-to-nearest-even, saturating to +-448, of the
 *    fp32 quotient float(x) / scale. E4M3 (OCP 8-bit floating point
 *    specification): 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent
 *    field 0 is subnormal (m * 2^-9); S.1111.111 is NaN; no infinities; the
 *    largest finite magnitude is 1.75 * 2^8 = 448.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - query head h reads KV head h / G with G = num_q_heads / num_kv_heads
 *    (contiguous groups);
 *  - split s of a request covers blocks [s*c, (s+1)*c) of its table, clipped
 *    to its own block count, with one chunk size c = ceil(n_max / S) for the
 *    whole batch, n_max = ceil(max_context_len / block_size); an empty split
 *    gives o = 0, lse = -inf;
 *  - a merge whose partials are all empty gives o = 0, lse = -inf.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Exact widening of a bf16 bit pattern: bf16 is the upper half of an fp32. */
double kfo_bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Offset of element (block, slot, kv_head, 0) in a [num_blocks, block_size,
 * num_kv_heads, head_dim] cache. */
static int64_t cache_row(int64_t block, int64_t slot, int kv_head,
                         int block_size, int num_kv_heads, int head_dim)
{
    return ((block * block_size + slot) * num_kv_heads + kv_head) * (int64_t)head_dim;
}

/* Token range of split `split` (reading above). Writes [*t_begin, *t_end). */
void kfo_split_range(int64_t ctx_len, int block_size, int num_splits,
                     int64_t max_context_len, int split,
                     int64_t *t_begin, int64_t *t_end)
{
    int64_t n_max = (max_context_len + block_size - 1) / block_size;
    int64_t chunk = (n_max + num_splits - 1) / num_splits;
    if (chunk < 1)
        chunk = 1;
    int64_t lo = (int64_t)split * chunk * block_size;
    int64_t hi = lo + chunk * block_size;
    if (lo > ctx_len)
        lo = ctx_len;
    if (hi > ctx_len)
        hi = ctx_len;
    *t_begin = lo;
    *t_end = hi;
}

/*
 * Attention of one query row over tokens [t_begin, t_end) of one request:
 *   s_t = scale * sum_d q[d] K_t[d]
 *   m   = max_t s_t,   l = sum_t e^{s_t - m}
 *   o   = sum_t e^{s_t - m} V_t / l,   lse = m + ln l
 * Empty range: o = 0, lse = -inf. Returns -1 (and writes nothing useful) if a
 * block id read from the table is outside [0, num_blocks).
 */
int kfo_partial(const uint16_t *q_row, const uint16_t *k_cache, const uint16_t *v_cache,
                const int32_t *bt_row, int64_t num_blocks, int block_size,
                int num_kv_heads, int head_dim, int kv_head,
                int64_t t_begin, int64_t t_end, double scale, double *o, double *lse)
{
    for (int d = 0; d < head_dim; ++d)
        o[d] = 0.0;
    if (t_end <= t_begin) {
        *lse = -INFINITY;
        return 0;
    }
    int64_t n = t_end - t_begin;
    double *s = (double *)malloc((size_t)n * sizeof(double));
    if (!s)
        return -2;

    /* scores */
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = t_begin + i;
        int64_t blk = bt_row[t / block_size];
        if (blk < 0 || blk >= num_blocks) {
            free(s);
            return -1;
        }
        const uint16_t *k = k_cache + cache_row(blk, t % block_size, kv_head,
                                                block_size, num_kv_heads, head_dim);
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += kfo_bf16_to_double(q_row[d]) * kfo_bf16_to_double(k[d]);
        s[i] = scale * dot;
        if (s[i] > m)
            m = s[i];
    }

    /* softmax weights and the weighted sum of values */
    double l = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = t_begin + i;
        int64_t blk = bt_row[t / block_size];
        const uint16_t *v = v_cache + cache_row(blk, t % block_size, kv_head,
                                                block_size, num_kv_heads, head_dim);
        double p = exp(s[i] - m);
        l += p;
        for (int d = 0; d < head_dim; ++d)
            o[d] += p * kfo_bf16_to_double(v[d]);
    }
    for (int d = 0; d < head_dim; ++d)
        o[d] /= l;
    *lse = m + log(l);
    free(s);
    return 0;
}

/*
 * LSE merge of `num_parts` partials (o_i normalised, lse_i):
 *   M = max_i lse_i,  w_i = e^{lse_i - M},
 *   o = sum_i w_i o_i / sum_i w_i,  lse = M + ln sum_i w_i.
 * Partial i is read at o_parts + i*o_stride and lse_parts[i*lse_stride].
 * A partial with lse = -inf has weight 0; if all are -inf, o = 0, lse = -inf.
 */
void kfo_merge(const double *o_parts, int64_t o_stride, const double *lse_parts,
               int64_t lse_stride, int num_parts, int head_dim, double *o, double *lse)
{
    double M = -INFINITY;
    for (int i = 0; i < num_parts; ++i) {
        double li = lse_parts[(int64_t)i * lse_stride];
        if (li > M)
            M = li;
    }
    for (int d = 0; d < head_dim; ++d)
        o[d] = 0.0;
    if (M == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double wsum = 0.0;
    for (int i = 0; i < num_parts; ++i) {
        double li = lse_parts[(int64_t)i * lse_stride];
        if (li == -INFINITY)
            continue;
        double w = exp(li - M);
        wsum += w;
        const double *oi = o_parts + (int64_t)i * o_stride;
        for (int d = 0; d < head_dim; ++d)
            o[d] += w * oi[d];
    }
    for (int d = 0; d < head_dim; ++d)
        o[d] /= wsum;
    *lse = M + log(wsum);
}

/* ------------------------------------------------------------------------- */
/* Batch drivers: all (request, query head) rows, or a listed subset, spread  */
/* over threads. Each row is independent; no blocking or reordering of the    */
/* arithmetic inside a row.                                                   */
/* ------------------------------------------------------------------------- */

typedef struct {
    const uint16_t *q, *k, *v;
    const int32_t *bt, *ctx;
    int bt_stride, batch, hq, hkv, d, bs, num_splits;
    int64_t num_blocks, max_ctx;
    double scale;
    const int32_t *rows; /* [n_rows][2] = (b, h) or NULL for all */
    int64_t n_rows;
    double *o_part, *lse_part;
    int n_threads, tid;
    int err;
} partial_job;

static void *partial_worker(void *arg)
{
    partial_job *j = (partial_job *)arg;
    int G = j->hq / j->hkv;
    for (int64_t r = j->tid; r < j->n_rows; r += j->n_threads) {
        int b, h;
        if (j->rows) {
            b = j->rows[2 * r];
            h = j->rows[2 * r + 1];
        } else {
            b = (int)(r / j->hq);
            h = (int)(r % j->hq);
        }
        const uint16_t *q_row = j->q + ((int64_t)b * j->hq + h) * j->d;
        const int32_t *bt_row = j->bt + (int64_t)b * j->bt_stride;
        for (int s = 0; s < j->num_splits; ++s) {
            int64_t t0, t1;
            kfo_split_range(j->ctx[b], j->bs, j->num_splits, j->max_ctx, s, &t0, &t1);
            int64_t slot = ((int64_t)s * j->batch + b) * j->hq + h;
            int rc = kfo_partial(q_row, j->k, j->v, bt_row, j->num_blocks, j->bs, j->hkv, j->d,
                                 h / G, t0, t1, j->scale, j->o_part + slot * j->d,
                                 j->lse_part + slot);
            if (rc != 0)
                j->err = rc;
        }
    }
    return NULL;
}

/*
 * Partials of every split for the listed rows (or all rows):
 *   o_part   [num_splits, batch, num_q_heads, head_dim]  (fp64)
 *   lse_part [num_splits, batch, num_q_heads]            (fp64)
 * Returns 0, -1 on a bad block id, -3 on a context length that is negative,
 * above the table capacity or above max_context_len, -4 on bad shapes.
 */
int kfo_decode_partials(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *block_tables, int bt_stride, const int32_t *ctx_lens,
                        int batch, int num_q_heads, int num_kv_heads, int head_dim,
                        int block_size, int64_t num_blocks, double scale, int num_splits,
                        int64_t max_context_len, const int32_t *rows, int64_t n_rows,
                        double *o_part, double *lse_part, int n_threads)
{
    if (num_splits < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0 || block_size < 1)
        return -4;
    for (int b = 0; b < batch; ++b)
        if (ctx_lens[b] < 0 || (int64_t)ctx_lens[b] > (int64_t)bt_stride * block_size ||
            ctx_lens[b] > max_context_len)
            return -3;
    if (!rows)
        n_rows = (int64_t)batch * num_q_heads;
    if (n_threads < 1)
        n_threads = 1;
    partial_job *jobs = (partial_job *)calloc((size_t)n_threads, sizeof(partial_job));
    pthread_t *th = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    for (int i = 0; i < n_threads; ++i) {
        partial_job *j = &jobs[i];
        j->q = q; j->k = k_cache; j->v = v_cache; j->bt = block_tables; j->ctx = ctx_lens;
        j->bt_stride = bt_stride; j->batch = batch; j->hq = num_q_heads; j->hkv = num_kv_heads;
        j->d = head_dim; j->bs = block_size; j->num_splits = num_splits;
        j->num_blocks = num_blocks; j->max_ctx = max_context_len; j->scale = scale;
        j->rows = rows; j->n_rows = n_rows; j->o_part = o_part; j->lse_part = lse_part;
        j->n_threads = n_threads; j->tid = i; j->err = 0;
    }
    if (n_threads == 1) {
        partial_worker(&jobs[0]);
    } else {
        for (int i = 0; i < n_threads; ++i)
            pthread_create(&th[i], NULL, partial_worker, &jobs[i]);
        for (int i = 0; i < n_threads; ++i)
            pthread_join(th[i], NULL);
    }
    int err = 0;
    for (int i = 0; i < n_threads; ++i)
        if (jobs[i].err)
            err = jobs[i].err;
    free(jobs);
    free(th);
    return err;
}

/*
 * Merge num_parts partial slots per row:
 *   o_part [num_parts, batch, num_q_heads, head_dim], lse_part [num_parts, batch, num_q_heads]
 *   out    [batch, num_q_heads, head_dim],            lse_out  [batch, num_q_heads]
 * Only the listed rows are written when `rows` is given.
 */
void kfo_merge_partials(const double *o_part, const double *lse_part, int num_parts,
                        int batch, int num_q_heads, int head_dim,
                        const int32_t *rows, int64_t n_rows, double *out, double *lse_out)
{
    if (!rows)
        n_rows = (int64_t)batch * num_q_heads;
    int64_t row_count = (int64_t)batch * num_q_heads;
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t row = rows ? (int64_t)rows[2 * r] * num_q_heads + rows[2 * r + 1] : r;
        kfo_merge(o_part + row * head_dim, row_count * head_dim, lse_part + row, row_count,
                  num_parts, head_dim, out + row * head_dim, lse_out + row);
    }
}

/*
 * Append: for each request b, position p = ctx_before[b] goes to block
 * block_tables[b][p / block_size], slot p % block_size; the K and V rows of
 * every KV head are copied there bit for bit. Every other element is left
 * as it was. Returns the number of requests skipped because the position or
 * the block id was out of range.
 */
int kfo_append(uint16_t *k_cache, uint16_t *v_cache, const uint16_t *k_new, const uint16_t *v_new,
               const int32_t *block_tables, int bt_stride, const int32_t *ctx_before,
               int batch, int num_kv_heads, int head_dim, int block_size, int64_t num_blocks)
{
    int skipped = 0;
    for (int b = 0; b < batch; ++b) {
        int64_t p = ctx_before[b];
        if (p < 0 || p >= (int64_t)bt_stride * block_size) {
            ++skipped;
            continue;
        }
        int64_t blk = block_tables[(int64_t)b * bt_stride + p / block_size];
        if (blk < 0 || blk >= num_blocks) {
            ++skipped;
            continue;
        }
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t dst = cache_row(blk, p % block_size, h, block_size, num_kv_heads, head_dim);
            int64_t src = ((int64_t)b * num_kv_heads + h) * head_dim;
            memcpy(k_cache + dst, k_new + src, (size_t)head_dim * sizeof(uint16_t));
            memcpy(v_cache + dst, v_new + src, (size_t)head_dim * sizeof(uint16_t));
        }
    }
    return skipped;
}

/* ------------------------------------------------------------------------- */
/* FP8 (E4M3) KV cache                                                        */
/* ------------------------------------------------------------------------- */

/* Value of an E4M3 code (NaN for S.1111.111). */
double kfo_e4m3_to_double(uint8_t code)
{
    int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);              /* subnormal: m/8 * 2^-6 */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* E4M3 code of x: round to nearest, ties to even, saturating to +-448; NaN -> 0x7F. */
uint8_t kfo_e4m3_from_float(float xf)
{
    double x = (double)xf;
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0)
        return sign | 0x7E;
    /* quantum of the binade holding a: 2^-9 below 2^-6, else 2^(e-3) */
    int e = a > 0 ? (int)floor(log2(a)) : -7;
    if (e < -6)
        e = -6;
    double quantum = ldexp(1.0, e - 3);
    double q = a / quantum;                  /* exact: a power-of-two scaling */
    double fl = floor(q);
    double frac = q - fl;
    double n = fl;
    if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) == 1.0))
        n = fl + 1.0;
    /* n in [0, 16]: back to exponent/mantissa fields */
    double v = n * quantum;
    if (v >= 448.0)
        return sign | 0x7E;
    if (v == 0.0)
        return sign;
    int ev = (int)floor(log2(v));
    if (ev < -6) {                           /* subnormal: v = m * 2^-9 */
        return sign | (uint8_t)(v / ldexp(1.0, -9));
    }
    int mant = (int)(v / ldexp(1.0, ev - 3)) - 8;
    return sign | (uint8_t)(((ev + 7) << 3) | mant);
}

/* Offset helper for a byte cache [num_blocks, block_size, num_kv_heads, head_dim]. */
static int64_t cache_row8(int64_t block, int64_t slot, int kv_head,
                          int block_size, int num_kv_heads, int head_dim)
{
    return ((block * block_size + slot) * num_kv_heads + kv_head) * (int64_t)head_dim;
}

/*
 * Attention of one query row over tokens [t_begin, t_end) of an FP8 cache:
 * the same definition as kfo_partial with K_t = decode(k code) * k_scale and
 * V_t = decode(v code) * v_scale (the scales of this KV head).
 */
int kfo_partial_fp8(const uint16_t *q_row, const uint8_t *k_cache, const uint8_t *v_cache,
                    double k_scale, double v_scale, const int32_t *bt_row, int64_t num_blocks,
                    int block_size, int num_kv_heads, int head_dim, int kv_head,
                    int64_t t_begin, int64_t t_end, double scale, double *o, double *lse)
{
    for (int d = 0; d < head_dim; ++d)
        o[d] = 0.0;
    if (t_end <= t_begin) {
        *lse = -INFINITY;
        return 0;
    }
    int64_t n = t_end - t_begin;
    double *s = (double *)malloc((size_t)n * sizeof(double));
    if (!s)
        return -2;
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = t_begin + i;
        int64_t blk = bt_row[t / block_size];
        if (blk < 0 || blk >= num_blocks) {
            free(s);
            return -1;
        }
        const uint8_t *k = k_cache + cache_row8(blk, t % block_size, kv_head, block_size,
                                                num_kv_heads, head_dim);
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += kfo_bf16_to_double(q_row[d]) * (kfo_e4m3_to_double(k[d]) * k_scale);
        s[i] = scale * dot;
        if (s[i] > m)
            m = s[i];
    }
    double l = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = t_begin + i;
        int64_t blk = bt_row[t / block_size];
        const uint8_t *v = v_cache + cache_row8(blk, t % block_size, kv_head, block_size,
                                                num_kv_heads, head_dim);
        double p = exp(s[i] - m);
        l += p;
        for (int d = 0; d < head_dim; ++d)
            o[d] += p * (kfo_e4m3_to_double(v[d]) * v_scale);
    }
    for (int d = 0; d < head_dim; ++d)
        o[d] /= l;
    *lse = m + log(l);
    free(s);
    return 0;
}

/* Partials of every split over an FP8 cache (see kfo_decode_partials);
 * k_scale, v_scale are fp32 [num_kv_heads]. Single-threaded. */
int kfo_decode_partials_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                            const float *k_scale, const float *v_scale,
                            const int32_t *block_tables, int bt_stride, const int32_t *ctx_lens,
                            int batch, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int64_t num_blocks, double scale, int num_splits,
                            int64_t max_context_len, const int32_t *rows, int64_t n_rows,
                            double *o_part, double *lse_part)
{
    if (num_splits < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0 || block_size < 1)
        return -4;
    for (int b = 0; b < batch; ++b)
        if (ctx_lens[b] < 0 || (int64_t)ctx_lens[b] > (int64_t)bt_stride * block_size ||
            ctx_lens[b] > max_context_len)
            return -3;
    int G = num_q_heads / num_kv_heads;
    if (!rows)
        n_rows = (int64_t)batch * num_q_heads;
    for (int64_t r = 0; r < n_rows; ++r) {
        int b = rows ? rows[2 * r] : (int)(r / num_q_heads);
        int h = rows ? rows[2 * r + 1] : (int)(r % num_q_heads);
        const uint16_t *q_row = q + ((int64_t)b * num_q_heads + h) * head_dim;
        const int32_t *bt_row = block_tables + (int64_t)b * bt_stride;
        int kvh = h / G;
        for (int s = 0; s < num_splits; ++s) {
            int64_t t0, t1;
            kfo_split_range(ctx_lens[b], block_size, num_splits, max_context_len, s, &t0, &t1);
            int64_t slot = ((int64_t)s * batch + b) * num_q_heads + h;
            int rc = kfo_partial_fp8(q_row, k_cache, v_cache, (double)k_scale[kvh],
                                     (double)v_scale[kvh], bt_row, num_blocks, block_size,
                                     num_kv_heads, head_dim, kvh, t0, t1, scale,
                                     o_part + slot * head_dim, lse_part + slot);
            if (rc != 0)
                return rc;
        }
    }
    return 0;
}

/*
 * FP8 append: request b's new bf16 K/V rows are quantised (code of
 * float(x) / scale[h], fp32 division) and written at position ctx_before[b]
 * as kfo_append does. Returns the number of requests skipped.
 */
int kfo_append_fp8(uint8_t *k_cache, uint8_t *v_cache, const uint16_t *k_new, const uint16_t *v_new,
                   const float *k_scale, const float *v_scale, const int32_t *block_tables,
                   int bt_stride, const int32_t *ctx_before, int batch, int num_kv_heads,
                   int head_dim, int block_size, int64_t num_blocks)
{
    int skipped = 0;
    for (int b = 0; b < batch; ++b) {
        int64_t p = ctx_before[b];
        if (p < 0 || p >= (int64_t)bt_stride * block_size) {
            ++skipped;
            continue;
        }
        int64_t blk = block_tables[(int64_t)b * bt_stride + p / block_size];
        if (blk < 0 || blk >= num_blocks) {
            ++skipped;
            continue;
        }
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t dst = cache_row8(blk, p % block_size, h, block_size, num_kv_heads, head_dim);
            int64_t src = ((int64_t)b * num_kv_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d) {
                float kq = (float)kfo_bf16_to_double(k_new[src + d]) / k_scale[h];
                float vq = (float)kfo_bf16_to_double(v_new[src + d]) / v_scale[h];
                k_cache[dst + d] = kfo_e4m3_from_float(kq);
                v_cache[dst + d] = kfo_e4m3_from_float(vq);
            }
        }
    }
    return skipped;
}

/* ------------------------------------------------------------------------- */
/* Multi-query (chunked prefill / shared prefix) attention                    */
/* ------------------------------------------------------------------------- */

/*
 * Partials for query tokens grouped by request: request b owns query rows
 * q_start[b] .. q_start[b+1]-1 (C_b of them) of q [num_q_tokens, Hq, D] and a
 * context of L_b = ctx_lens[b] cached tokens (the chunk included). Query j of
 * request b attends tokens [0, limit) with limit = L_b - C_b + j + 1 if causal,
 * L_b otherwise; split s keeps the part of its token range (the decode split
 * rule) below the limit. Writes o_part [S, num_q_tokens, Hq, D] and
 * lse_part [S, num_q_tokens, Hq]. Returns -3 on C_b > L_b (causal) or a bad
 * length, -1 on a bad block id.
 */
int kfo_multiquery_partials(const uint16_t *q, const int32_t *q_start, const uint16_t *k_cache,
                            const uint16_t *v_cache, const int32_t *block_tables, int bt_stride,
                            const int32_t *ctx_lens, int causal, int batch, int num_q_tokens,
                            int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            int64_t num_blocks, double scale, int num_splits,
                            int64_t max_context_len, double *o_part, double *lse_part)
{
    if (num_splits < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0 || block_size < 1)
        return -4;
    int G = num_q_heads / num_kv_heads;
    for (int b = 0; b < batch; ++b) {
        int64_t L = ctx_lens[b];
        int64_t C = (int64_t)q_start[b + 1] - q_start[b];
        if (L < 0 || L > (int64_t)bt_stride * block_size || L > max_context_len || C < 0 ||
            q_start[b + 1] > num_q_tokens || (causal && C > L))
            return -3;
        const int32_t *bt_row = block_tables + (int64_t)b * bt_stride;
        for (int64_t j = 0; j < C; ++j) {
            int64_t n = q_start[b] + j;
            int64_t limit = causal ? L - C + j + 1 : L;
            for (int h = 0; h < num_q_heads; ++h) {
                const uint16_t *q_row = q + (n * num_q_heads + h) * head_dim;
                for (int s = 0; s < num_splits; ++s) {
                    int64_t t0, t1;
                    kfo_split_range(L, block_size, num_splits, max_context_len, s, &t0, &t1);
                    if (t1 > limit)
                        t1 = limit;
                    if (t0 > t1)
                        t0 = t1;
                    int64_t slot = ((int64_t)s * num_q_tokens + n) * num_q_heads + h;
                    int rc = kfo_partial(q_row, k_cache, v_cache, bt_row, num_blocks, block_size,
                                         num_kv_heads, head_dim, h / G, t0, t1, scale,
                                         o_part + slot * head_dim, lse_part + slot);
                    if (rc != 0)
                        return rc;
                }
            }
        }
    }
    return 0;
}

