/*
 * oracle.c -- plain, slow, fp64 CPU definition of one continuous-batching
 * attention step over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the parity oracle: only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or helper with the CUDA library; the
 * product path never calls it.
 *
 * Every function below computes the plain definition of its operation, one
 * element at a time, in double precision, from the same bf16 bit patterns the
 * GPU reads.  No blocking, fusion or reordering beyond the definition.
 *
 * Sources (web pages on vLLM-style serving):
 *  [TC]  "vLLM中如何实现大模型推理加速技术？" (cloud.tencent.com.cn, article
 *        2589754): 90-token concatenated prefill (31/29/30); chunked prefill
 *        (48 = 16+16+16, later chunks attend to cached KV, offset mask);
 *        prefix-cache hit (107 tokens, 48 cached, positions from 48);
 *        speculative verify (1 + N draft tokens in one pass).
 *  [CH]  "11. 推理加速(一):vLLM 原理" (chuoer47.github.io): §11.2 PagedAttention
 *        (fixed-size blocks, per-request block table, shared blocks
 *        [3,7,11] vs [3,7,5]); §11.3 prefill vs decode.
 *  [AI]  2048ai.net page on the vLLM V1 engine, §02 推理优化 › 1. 级联推理
 *        (Cascade Inference): shared-prefix attention state + unique-suffix
 *        state combined by an associative, commutative merge operator.
 *
 * Readings where the pages are silent (all listed in the design notes):
 *  - cache layout [num_blocks][num_kv_heads][block_size][head_dim];
 *  - slot = physical_block * block_size + offset, negative slot = skip;
 *  - row i of a request with context c attends keys 0..c+i inclusive;
 *  - q head h uses kv head h / (num_q_heads / num_kv_heads);
 *  - attention state = (normalised output, natural-log sum-exp of the scaled
 *    scores); the empty state is (0, -inf).
 *
 * Parity pins: every function here is pinned by tests that do not call it
 * twice -- brute force on tiny inputs, torch's scaled_dot_product_attention
 * on the single-request case, closed forms, and the pages' worked examples.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_BAD_ARG 1
#define ORC_BAD_META 2
#define ORC_NO_MEM 3

/* bf16 is the top half of an IEEE binary32: widen exactly. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Cache element index of (physical block, kv head, offset in block, dim). */
static int64_t cache_index(int64_t blk, int64_t head, int64_t off, int64_t dim,
                           int32_t num_kv_heads, int32_t block_size, int32_t head_dim)
{
    return ((blk * num_kv_heads + head) * block_size + off) * head_dim + dim;
}

/*
 * FP8 KV cache (quantisation of the KV cache, [AI] §02 推理优化): elements are
 * stored as OCP FP8 E4M3 ("e4m3fn") codes with one fp32 scale per kv head for
 * K and one for V; an element's value is decode(code) * scale.
 *
 * E4M3 as defined by the format: sign bit, 4 exponent bits (bias 7), 3
 * mantissa bits.  Exponent field 0 holds the subnormals m/8 * 2^-6; fields
 * 1..15 hold (1 + m/8) * 2^(e-7), except S.1111.111, which is NaN.  There is
 * no infinity; the largest finite magnitude is 1.75 * 2^8 = 448.
 */
static double e4m3_value(uint8_t code)
{
    int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/*
 * Encoding (a reading: the pages name FP8 KV caches without fixing the
 * rounding): round to the nearest representable magnitude, ties to the even
 * mantissa, and saturate magnitudes beyond 448 (including infinity) to 448.
 * NaN encodes as 0x7F.
 */
static uint8_t e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal grid: multiples of 2^-9; a result of 8 * 2^-9 = 2^-6 is
         * the smallest normal, whose code (exponent 1, mantissa 0) is 8 too */
        double q = nearbyint(ldexp(a, 9)); /* default rounding: ties to even */
        return sign | (uint8_t)q;
    }
    int e = ilogb(a);                        /* 2^e <= a < 2^(e+1), -6 <= e <= 8 */
    double q = nearbyint(ldexp(a, 3 - e));   /* in [8, 16] */
    if (q == 16.0) {
        q = 8.0;
        e += 1;
    }
    if (e > 8 || (e == 8 && q > 14.0))
        return sign | 0x7E;
    return sign | (uint8_t)(((e + 7) << 3) | ((int)q - 8));
}

/* Array forms of the two conversions (pinned on their own by the tests). */
int oracle_e4m3_encode(const float *x, int64_t n, uint8_t *codes)
{
    if (n < 0)
        return ORC_BAD_ARG;
    for (int64_t i = 0; i < n; ++i)
        codes[i] = e4m3_encode(x[i]);
    return ORC_OK;
}

int oracle_e4m3_decode(const uint8_t *codes, int64_t n, double *x)
{
    if (n < 0)
        return ORC_BAD_ARG;
    for (int64_t i = 0; i < n; ++i)
        x[i] = e4m3_value(codes[i]);
    return ORC_OK;
}

/*
 * reshape_and_cache: for every new token t with slot s = slot_mapping[t] >= 0,
 * cache[s / block_size][h][s % block_size][:] = k[t][h][:] (same for v).
 * Pure bit copy.  [CH] §11.2 (a token lands in a slot of a fixed-size block).
 */
int oracle_write_kv(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping,
                    int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                    int32_t block_size, int32_t num_blocks,
                    uint16_t *k_cache, uint16_t *v_cache)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0)
        return ORC_BAD_ARG;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s < 0)
            continue;
        int64_t blk = s / block_size;
        int64_t off = s % block_size;
        if (blk >= num_blocks)
            return ORC_BAD_META;
        for (int64_t h = 0; h < num_kv_heads; ++h) {
            for (int64_t e = 0; e < head_dim; ++e) {
                int64_t src = (t * num_kv_heads + h) * head_dim + e;
                int64_t dst = cache_index(blk, h, off, e, num_kv_heads, block_size, head_dim);
                k_cache[dst] = k[src];
                v_cache[dst] = v[src];
            }
        }
    }
    return ORC_OK;
}

/*
 * reshape_and_cache into an FP8 cache: the same slots as oracle_write_kv,
 * each element stored as e4m3_encode(x / scale[h]), the quotient taken in
 * binary32 (x is the bf16 value widened exactly; the division rounds to
 * nearest even), then encoded as above.
 */
int oracle_write_kv_fp8(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping,
                        int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                        int32_t block_size, int32_t num_blocks, const float *k_scale,
                        const float *v_scale, uint8_t *k_cache, uint8_t *v_cache)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0)
        return ORC_BAD_ARG;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s < 0)
            continue;
        int64_t blk = s / block_size;
        int64_t off = s % block_size;
        if (blk >= num_blocks)
            return ORC_BAD_META;
        for (int64_t h = 0; h < num_kv_heads; ++h) {
            for (int64_t e = 0; e < head_dim; ++e) {
                int64_t src = (t * num_kv_heads + h) * head_dim + e;
                int64_t dst = cache_index(blk, h, off, e, num_kv_heads, block_size, head_dim);
                float kx = (float)bf16_value(k[src]), vx = (float)bf16_value(v[src]);
                float kq = kx / k_scale[h], vq = vx / v_scale[h];
                k_cache[dst] = e4m3_encode(kq);
                v_cache[dst] = e4m3_encode(vq);
            }
        }
    }
    return ORC_OK;
}

/*
 * One query row against `nkeys` gathered keys, of which the first `visible`
 * are attended (visible <= nkeys).  Writes the normalised output and the
 * natural-log sum-exp of the scaled scores.  scores/tmp are scratch.
 */
static void attend_row(const double *qrow, const double *keys, const double *vals,
                       int64_t visible, int32_t head_dim, double scale,
                       double *scores, double *out_row, double *lse_out)
{
    if (visible <= 0) {
        for (int32_t e = 0; e < head_dim; ++e)
            out_row[e] = 0.0;
        *lse_out = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < visible; ++j) {
        double dot = 0.0;
        for (int32_t e = 0; e < head_dim; ++e)
            dot += qrow[e] * keys[j * head_dim + e];
        scores[j] = scale * dot;
        if (scores[j] > m)
            m = scores[j];
    }
    double sum = 0.0;
    for (int64_t j = 0; j < visible; ++j)
        sum += exp(scores[j] - m);
    double lse = m + log(sum);
    for (int32_t e = 0; e < head_dim; ++e)
        out_row[e] = 0.0;
    for (int64_t j = 0; j < visible; ++j) {
        double p = exp(scores[j] - lse);
        for (int32_t e = 0; e < head_dim; ++e)
            out_row[e] += p * vals[j * head_dim + e];
    }
    *lse_out = lse;
}

/* The caches of one call: bf16 bit patterns, or e4m3 codes with per-kv-head
 * scales. */
typedef struct {
    const void *k, *v;
    const float *k_scale, *v_scale; /* fp8 only */
    int fp8;
} kv_source;

static double kv_element(const kv_source *src, int is_v, int64_t idx, int32_t head)
{
    if (!src->fp8)
        return bf16_value(((const uint16_t *)(is_v ? src->v : src->k))[idx]);
    uint8_t code = ((const uint8_t *)(is_v ? src->v : src->k))[idx];
    return e4m3_value(code) * (double)(is_v ? src->v_scale[head] : src->k_scale[head]);
}

/* Gather keys [0, len) of one kv head through a block table into dense
 * [len][head_dim] arrays.  [CH] §11.2: logical block j -> physical block. */
static int gather_kv(const kv_source *src, const int32_t *table_row, int64_t len, int32_t head,
                     int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                     int32_t head_dim, double *keys, double *vals)
{
    for (int64_t j = 0; j < len; ++j) {
        int64_t blk = table_row[j / block_size];
        int64_t off = j % block_size;
        if (blk < 0 || blk >= num_blocks)
            return ORC_BAD_META;
        for (int32_t e = 0; e < head_dim; ++e) {
            int64_t idx = cache_index(blk, head, off, e, num_kv_heads, block_size, head_dim);
            keys[j * head_dim + e] = kv_element(src, 0, idx, head);
            vals[j * head_dim + e] = kv_element(src, 1, idx, head);
        }
    }
    return ORC_OK;
}

/*
 * Varlen causal attention for one step.  Request b owns query tokens
 * [qsl[b], qsl[b+1]); its first context_lens[b] tokens are already cached and
 * seq_lens[b] = context_lens[b] + q_len.  Row i (absolute position
 * context + i, [TC] prefix-cache example: positions start after the hit)
 * attends keys 0..context+i ([TC] chunked prefill: later chunks see all
 * cached KV plus their own causal triangle).  Keys are read through
 * block_tables[b] ([CH] §11.2).
 *
 * out: double [num_q_tokens][num_q_heads][head_dim]; lse: double
 * [num_q_tokens][num_q_heads]; visible (optional): int32 [num_q_tokens], the
 * number of keys each row attends to.
 */
static int attention_impl(const uint16_t *q, const kv_source *src,
                          int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                          int32_t head_dim, const int32_t *block_tables,
                          int32_t max_blocks_per_seq, const int32_t *query_start_loc,
                          const int32_t *context_lens, const int32_t *seq_lens, int32_t num_seqs,
                          int32_t num_q_heads, double scale, double *out, double *lse,
                          int32_t *visible)
{
    if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_q_heads % num_kv_heads != 0)
        return ORC_BAD_ARG;
    const int32_t group = num_q_heads / num_kv_heads;
    for (int32_t b = 0; b < num_seqs; ++b) {
        int64_t n = (int64_t)query_start_loc[b + 1] - query_start_loc[b];
        if (n < 0 || context_lens[b] < 0 || (int64_t)seq_lens[b] != context_lens[b] + n)
            return ORC_BAD_META;
        if (((int64_t)seq_lens[b] + block_size - 1) / block_size > max_blocks_per_seq)
            return ORC_BAD_META;
    }
    int status = ORC_OK;
    /* One task per (request, kv head). */
    const int64_t ntask = (int64_t)num_seqs * num_kv_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t task = 0; task < ntask; ++task) {
        int32_t b = (int32_t)(task / num_kv_heads);
        int32_t hk = (int32_t)(task % num_kv_heads);
        int64_t n = (int64_t)query_start_loc[b + 1] - query_start_loc[b];
        int64_t ctx = context_lens[b];
        int64_t len = seq_lens[b];
        if (n == 0)
            continue;
        double *keys = (double *)malloc(sizeof(double) * (size_t)(len * head_dim + 1));
        double *vals = (double *)malloc(sizeof(double) * (size_t)(len * head_dim + 1));
        double *scores = (double *)malloc(sizeof(double) * (size_t)(len + 1));
        double *qrow = (double *)malloc(sizeof(double) * (size_t)head_dim);
        if (!keys || !vals || !scores || !qrow) {
#pragma omp atomic write
            status = ORC_NO_MEM;
            free(keys); free(vals); free(scores); free(qrow);
            continue;
        }
        const int32_t *table_row = block_tables + (int64_t)b * max_blocks_per_seq;
        if (gather_kv(src, table_row, len, hk, num_blocks, block_size,
                      num_kv_heads, head_dim, keys, vals) != ORC_OK) {
#pragma omp atomic write
            status = ORC_BAD_META;
            free(keys); free(vals); free(scores); free(qrow);
            continue;
        }
        for (int64_t i = 0; i < n; ++i) {
            int64_t t = query_start_loc[b] + i;
            int64_t position = ctx + i;
            int64_t nvis = position + 1; /* keys 0..position inclusive */
            if (nvis > len)
                nvis = len;
            if (visible && hk == 0)
                visible[t] = (int32_t)nvis;
            for (int32_t j = 0; j < group; ++j) {
                int32_t h = hk * group + j;
                for (int32_t e = 0; e < head_dim; ++e)
                    qrow[e] = bf16_value(q[(t * num_q_heads + h) * head_dim + e]);
                attend_row(qrow, keys, vals, nvis, head_dim, scale, scores,
                           out + (t * num_q_heads + h) * head_dim,
                           lse + t * num_q_heads + h);
            }
        }
        free(keys); free(vals); free(scores); free(qrow);
    }
    return status;
}

int oracle_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                     int32_t num_blocks, int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                     const int32_t *block_tables, int32_t max_blocks_per_seq,
                     const int32_t *query_start_loc, const int32_t *context_lens,
                     const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
                     double scale, double *out, double *lse, int32_t *visible)
{
    kv_source src = {k_cache, v_cache, NULL, NULL, 0};
    return attention_impl(q, &src, num_blocks, block_size, num_kv_heads, head_dim, block_tables,
                          max_blocks_per_seq, query_start_loc, context_lens, seq_lens, num_seqs,
                          num_q_heads, scale, out, lse, visible);
}

/* The same attention over an FP8 cache: every key and value element is
 * decode(code) * scale[kv head], in fp64, before the plain definition. */
int oracle_attention_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                         const float *k_scale, const float *v_scale, int32_t num_blocks,
                         int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                         const int32_t *block_tables, int32_t max_blocks_per_seq,
                         const int32_t *query_start_loc, const int32_t *context_lens,
                         const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
                         double scale, double *out, double *lse, int32_t *visible)
{
    kv_source src = {k_cache, v_cache, k_scale, v_scale, 1};
    return attention_impl(q, &src, num_blocks, block_size, num_kv_heads, head_dim, block_tables,
                          max_blocks_per_seq, query_start_loc, context_lens, seq_lens, num_seqs,
                          num_q_heads, scale, out, lse, visible);
}

/*
 * Shared-prefix ("multi-query") attention of cascade inference ([AI] §02.1):
 * every query row of every request attends all prefix_len keys listed by
 * prefix_blocks, with no mask (the prefix precedes every query position).
 * out/lse as in oracle_attention, one state per (token, q head).
 */
int oracle_prefix_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                            int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                            int32_t head_dim, const int32_t *prefix_blocks, int32_t prefix_len,
                            int32_t num_q_tokens, int32_t num_q_heads, double scale,
                            double *out, double *lse)
{
    if (num_q_tokens < 0 || prefix_len < 0 || num_kv_heads <= 0 || num_q_heads <= 0 ||
        head_dim <= 0 || block_size <= 0 || num_q_heads % num_kv_heads != 0)
        return ORC_BAD_ARG;
    const int32_t group = num_q_heads / num_kv_heads;
    int status = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t hk = 0; hk < num_kv_heads; ++hk) {
        double *keys = (double *)malloc(sizeof(double) * (size_t)((int64_t)prefix_len * head_dim + 1));
        double *vals = (double *)malloc(sizeof(double) * (size_t)((int64_t)prefix_len * head_dim + 1));
        double *scores = (double *)malloc(sizeof(double) * (size_t)(prefix_len + 1));
        double *qrow = (double *)malloc(sizeof(double) * (size_t)head_dim);
        if (!keys || !vals || !scores || !qrow) {
#pragma omp atomic write
            status = ORC_NO_MEM;
            free(keys); free(vals); free(scores); free(qrow);
            continue;
        }
        kv_source src = {k_cache, v_cache, NULL, NULL, 0};
        if (gather_kv(&src, prefix_blocks, prefix_len, hk, num_blocks, block_size,
                      num_kv_heads, head_dim, keys, vals) != ORC_OK) {
#pragma omp atomic write
            status = ORC_BAD_META;
            free(keys); free(vals); free(scores); free(qrow);
            continue;
        }
        for (int64_t t = 0; t < num_q_tokens; ++t) {
            for (int32_t j = 0; j < group; ++j) {
                int32_t h = hk * group + j;
                for (int32_t e = 0; e < head_dim; ++e)
                    qrow[e] = bf16_value(q[(t * num_q_heads + h) * head_dim + e]);
                attend_row(qrow, keys, vals, prefix_len, head_dim, scale, scores,
                           out + (t * num_q_heads + h) * head_dim, lse + t * num_q_heads + h);
            }
        }
        free(keys); free(vals); free(scores); free(qrow);
    }
    return status;
}

/*
 * Merge operator of cascade inference ([AI] §02.1): two attention states over
 * disjoint key sets combine into the state over their union.
 *   lse = M + ln(e^(lse_a - M) + e^(lse_b - M)),  M = max(lse_a, lse_b)
 *   o   = e^(lse_a - lse) o_a + e^(lse_b - lse) o_b
 * Two empty states (lse = -inf) give the empty state (0, -inf).
 * o_*: double [n][num_heads][head_dim]; lse_*: double [n][num_heads].
 */
int oracle_merge_states(const double *o_a, const double *lse_a, const double *o_b,
                        const double *lse_b, int64_t n, int32_t num_heads, int32_t head_dim,
                        double *out, double *lse_out)
{
    if (n < 0 || num_heads <= 0 || head_dim <= 0)
        return ORC_BAD_ARG;
    for (int64_t r = 0; r < n * num_heads; ++r) {
        double la = lse_a[r], lb = lse_b[r];
        double m = la > lb ? la : lb;
        if (m == -INFINITY) {
            for (int32_t e = 0; e < head_dim; ++e)
                out[r * head_dim + e] = 0.0;
            lse_out[r] = -INFINITY;
            continue;
        }
        double l = m + log(exp(la - m) + exp(lb - m));
        double wa = exp(la - l), wb = exp(lb - l);
        for (int32_t e = 0; e < head_dim; ++e)
            out[r * head_dim + e] = wa * o_a[r * head_dim + e] + wb * o_b[r * head_dim + e];
        lse_out[r] = l;
    }
    return ORC_OK;
}
