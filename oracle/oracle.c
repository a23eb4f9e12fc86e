/*
 * oracle.c -- plain, slow CPU statement of paged decode attention and of the
 * slot-mapped KV append, in IEEE double.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path includes, links or
 * calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or table with the CUDA
 * library: it decodes and encodes IEEE binary16 itself.
 *
 * Sources (page title, section):
 *  - "Distributed LLM Inference Serving Platform", section 2 (Mental Model):
 *    a sequence's KV cache is cut into fixed-size logical blocks of e.g. 16
 *    tokens; a block table maps each logical block number to a physical block
 *    of the HBM pool, like an OS page table.
 *  - same page, section 3 (PagedAttention row): the attention kernel reads
 *    K and V vectors from non-contiguous physical blocks through that table.
 *  - same page, section 5.1 (Continuous Decode Loop): each decode step, every
 *    active sequence attends with its newest token over all previous blocks
 *    in its block table; new K/V vectors are written into the assigned
 *    physical blocks (Chunked Prefill item, "Allocate 1 token page" arrow).
 *  - same page, section 1 (KV Cache Memory Explosion) and the Lab 3 roofline
 *    listing's nHeads / nKvHeads parameters: grouped-query attention, several
 *    query heads share one KV head (8:1 for the 70B model).
 *  - softmax(q K^T * scale) V is the attention the FlashAttention-2 paper
 *    (cited in section 14 of that page) computes; its log-sum-exp merge of
 *    partial results is the flash-decoding split.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - cache layout [num_blocks][n_kv_heads][block_size][head_dim], fp16;
 *  - slot = physical_block * block_size + offset, int64; slot < 0 = padding;
 *  - query head h reads KV head h / (n_q_heads / n_kv_heads);
 *  - context_lens[b] = number of tokens attended, positions [0, L);
 *  - L = 0 gives out = 0 and lse = -inf;
 *  - a block id outside [0, num_blocks) among the first ceil(L/bs) table
 *    entries makes the input invalid: the oracle rejects it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------------
 * IEEE 754 binary16 <-> double.
 * binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * ------------------------------------------------------------------------- */

double pkvo_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);                 /* zero or subnormal */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25);  /* (1.frac) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Round-to-nearest-even encode.  Scaling by a power of two is exact in
 * double, so rint() (round-half-even in the default rounding mode) performs
 * the one rounding step. */
uint16_t pkvo_f64_to_f16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7e00);
    if (isinf(a)) return (uint16_t)(sign | 0x7c00);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: value = m * 2^-24, m in [0, 1024]; m == 1024 is
         * the smallest normal number, whose bit pattern is 0x0400 */
        double m = rint(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)m);
    }
    int e2;
    frexp(a, &e2);                    /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;                   /* a in [2^e, 2^(e+1)) */
    double m = rint(ldexp(a, 10 - e)); /* 11-bit significand, in [1024, 2048] */
    if (m == 2048.0) { m = 1024.0; e += 1; }
    if (e > 15) return (uint16_t)(sign | 0x7c00);   /* overflow -> inf */
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)((int)m - 1024));
}

/* Lookup table of all 65536 decoded values: the same function, evaluated
 * once per bit pattern, so that the loops below stay readable and finish. */
static double g_f16[65536];
static int g_f16_ready = 0;

static void f16_table_init(void)
{
    if (g_f16_ready) return;
    for (int i = 0; i < 65536; ++i) g_f16[i] = pkvo_f16_to_f64((uint16_t)i);
    g_f16_ready = 1;
}

void pkvo_init(void) { f16_table_init(); }

/* ---------------------------------------------------------------------------
 * Slot-mapped append.  For token i and KV head j the new K (and V) vector is
 * written into the physical block slot_mapping[i] / block_size at row
 * slot_mapping[i] % block_size.  A negative slot marks a padding token and is
 * skipped.  Returns 0, or -1 if some slot lies beyond the pool (that token is
 * not written).
 * ------------------------------------------------------------------------- */
int pkvo_append(const uint16_t *k_new, const uint16_t *v_new, const int64_t *slot_mapping,
                uint16_t *k_cache, uint16_t *v_cache, int num_tokens, int n_kv_heads,
                int head_dim, int block_size, int64_t num_blocks)
{
    int rc = 0;
    for (int i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= num_blocks * (int64_t)block_size) { rc = -1; continue; }
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        for (int j = 0; j < n_kv_heads; ++j) {
            const uint16_t *ksrc = k_new + ((int64_t)i * n_kv_heads + j) * head_dim;
            const uint16_t *vsrc = v_new + ((int64_t)i * n_kv_heads + j) * head_dim;
            int64_t row = ((block * n_kv_heads + j) * block_size + offset) * head_dim;
            for (int k = 0; k < head_dim; ++k) {
                k_cache[row + k] = ksrc[k];
                v_cache[row + k] = vsrc[k];
            }
        }
    }
    return rc;
}

/* Address of logical token t of sequence b, KV head j, or NULL when the
 * block table entry is not a block of the pool. */
static const uint16_t *token_row(const uint16_t *cache, const int32_t *block_tables,
                                 int max_blocks_per_seq, int64_t num_blocks, int n_kv_heads,
                                 int head_dim, int block_size, int b, int j, int t)
{
    int32_t block = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];
    if (block < 0 || block >= num_blocks) return NULL;
    int64_t row = (((int64_t)block * n_kv_heads + j) * block_size + t % block_size) * head_dim;
    return cache + row;
}

/* Softmax attention of query head h of sequence b over the logical tokens
 * [t_begin, t_end).  Outputs, for that range:
 *   m   = max_t s_t                  (s_t = scale * q . K_t)
 *   l   = sum_t exp(s_t - m)
 *   acc = sum_t exp(s_t - m) V_t     (not normalised)
 * An empty range gives m = -inf, l = 0, acc = 0.  Returns 0, or -1 when a
 * block id in the range is invalid. */
static int attend_range(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *block_tables, int max_blocks_per_seq, int64_t num_blocks,
                        double scale, int n_q_heads, int n_kv_heads, int head_dim,
                        int block_size, int b, int h, int t_begin, int t_end,
                        double *m_out, double *l_out, double *acc)
{
    int group = n_q_heads / n_kv_heads;
    int j = h / group;                        /* KV head read by query head h */
    int n = t_end - t_begin;
    for (int k = 0; k < head_dim; ++k) acc[k] = 0.0;
    *m_out = -INFINITY;
    *l_out = 0.0;
    if (n <= 0) return 0;

    const uint16_t *qv = q + ((int64_t)b * n_q_heads + h) * head_dim;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    if (!s) return -2;

    /* step 1-2: gather K_t in logical order, logits in double */
    for (int t = t_begin; t < t_end; ++t) {
        const uint16_t *kt = token_row(k_cache, block_tables, max_blocks_per_seq, num_blocks,
                                       n_kv_heads, head_dim, block_size, b, j, t);
        if (!kt) { free(s); return -1; }
        double dot = 0.0;
        for (int k = 0; k < head_dim; ++k) dot += g_f16[qv[k]] * g_f16[kt[k]];
        s[t - t_begin] = scale * dot;
    }
    /* step 3: exponentials relative to the range maximum */
    double m = -INFINITY;
    for (int i = 0; i < n; ++i) if (s[i] > m) m = s[i];
    double l = 0.0;
    for (int i = 0; i < n; ++i) { s[i] = exp(s[i] - m); l += s[i]; }
    /* step 4: weighted sum of V_t */
    for (int t = t_begin; t < t_end; ++t) {
        const uint16_t *vt = token_row(v_cache, block_tables, max_blocks_per_seq, num_blocks,
                                       n_kv_heads, head_dim, block_size, b, j, t);
        double p = s[t - t_begin];
        for (int k = 0; k < head_dim; ++k) acc[k] += p * g_f16[vt[k]];
    }
    free(s);
    *m_out = m;
    *l_out = l;
    return 0;
}

/* ---------------------------------------------------------------------------
 * Decode attention for every (sequence b, query head h) with mask[b*H+h] != 0
 * (mask NULL = all).  out[b][h][:] = sum_t p_t V_t with p = softmax(s);
 * lse[b][h] = m + ln(l); out_f16 is the round-to-nearest-even fp16 copy.
 * Any of out / lse / out_f16 may be NULL.  num_threads <= 0 uses the OpenMP
 * default.  Returns 0, or -1 when an input is invalid (a bad block id, a
 * context length outside [0, max_blocks_per_seq*block_size], or n_q_heads
 * not a multiple of n_kv_heads).
 * ------------------------------------------------------------------------- */
int pkvo_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                int max_blocks_per_seq, int64_t num_blocks, double scale, int n_q_heads,
                int n_kv_heads, int head_dim, int block_size, const uint8_t *mask,
                double *out, double *lse, uint16_t *out_f16, int num_threads)
{
    f16_table_init();
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return -1;
    for (int b = 0; b < num_seqs; ++b) {
        int L = context_lens[b];
        if (L < 0 || L > max_blocks_per_seq * block_size) return -1;
    }
    int failed = 0;
    int64_t pairs = (int64_t)num_seqs * n_q_heads;
#ifdef _OPENMP
    int nt = num_threads > 0 ? num_threads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt) reduction(| : failed)
#endif
    for (int64_t bh = 0; bh < pairs; ++bh) {
        if (mask && !mask[bh]) continue;
        int b = (int)(bh / n_q_heads);
        int h = (int)(bh % n_q_heads);
        double *acc = (double *)malloc(sizeof(double) * (size_t)head_dim);
        double m, l;
        int rc = attend_range(q, k_cache, v_cache, block_tables, max_blocks_per_seq, num_blocks,
                              scale, n_q_heads, n_kv_heads, head_dim, block_size, b, h, 0,
                              context_lens[b], &m, &l, acc);
        if (rc != 0) { failed = 1; free(acc); continue; }
        for (int k = 0; k < head_dim; ++k) {
            double o = (l > 0.0) ? acc[k] / l : 0.0;
            if (out) out[bh * head_dim + k] = o;
            if (out_f16) out_f16[bh * head_dim + k] = pkvo_f64_to_f16(o);
        }
        if (lse) lse[bh] = (l > 0.0) ? m + log(l) : -INFINITY;
        free(acc);
    }
    (void)num_threads;
    return failed ? -1 : 0;
}

/* Partial result of one (b, h) over tokens [t_begin, t_end): (m, l, acc) as
 * defined for attend_range. */
int pkvo_decode_partial(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *block_tables, int max_blocks_per_seq, int64_t num_blocks,
                        double scale, int n_q_heads, int n_kv_heads, int head_dim,
                        int block_size, int b, int h, int t_begin, int t_end,
                        double *m_out, double *l_out, double *acc_out)
{
    f16_table_init();
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return -1;
    return attend_range(q, k_cache, v_cache, block_tables, max_blocks_per_seq, num_blocks,
                        scale, n_q_heads, n_kv_heads, head_dim, block_size, b, h, t_begin,
                        t_end, m_out, l_out, acc_out);
}

/* Log-sum-exp merge of n partial results (m_i, l_i, acc_i) that cover
 * disjoint token ranges of the same (b, h):
 *   M = max_i m_i,  out = sum_i e^(m_i-M) acc_i / sum_i e^(m_i-M) l_i,
 *   lse = M + ln(sum_i e^(m_i-M) l_i).
 * Empty partials (m = -inf) carry weight 0.  All empty: out = 0, lse = -inf. */
void pkvo_lse_merge(int n, const double *m, const double *l, const double *acc, int head_dim,
                    double *out, double *lse)
{
    double M = -INFINITY;
    for (int i = 0; i < n; ++i) if (m[i] > M) M = m[i];
    for (int k = 0; k < head_dim; ++k) out[k] = 0.0;
    if (M == -INFINITY) { *lse = -INFINITY; return; }
    double denom = 0.0;
    for (int i = 0; i < n; ++i) {
        if (m[i] == -INFINITY) continue;
        double w = exp(m[i] - M);
        denom += w * l[i];
        for (int k = 0; k < head_dim; ++k) out[k] += w * acc[(int64_t)i * head_dim + k];
    }
    for (int k = 0; k < head_dim; ++k) out[k] /= denom;
    *lse = M + log(denom);
}

/* ---------------------------------------------------------------------------
 * FP8 KV cache.  "Roadmap: vLLM-style serving features for TornadoVM batched
 * decode", KV-cache list: a quantized (Q8/FP8) KV cache is named as future
 * work, with no format or scaling rule.  Reading (listed in the design
 * notes): OCP FP8 E4M3 ("e4m3fn": 1 sign, 4 exponent bits with bias 7, 3
 * fraction bits, no infinities, S.1111.111 = NaN, largest finite 448), one
 * scale per cache tensor supplied by the caller.  A cached value is
 *     code = E4M3(y),  y = fp32(x) / fp32(scale)  (IEEE fp32 division),
 * with E4M3() rounding to nearest, ties to even, and saturating finite
 * overflow and infinities to +-448; a NaN gives the NaN code 0x7f.  The
 * attended value is decode(code) * scale.
 * ------------------------------------------------------------------------- */

double pkvo_e4m3_to_f64(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int expo = (c >> 3) & 15;
    int frac = c & 7;
    double v;
    if (expo == 15 && frac == 7) {
        v = NAN;
    } else if (expo == 0) {
        v = ldexp((double)frac, -9);                /* zero or subnormal: frac * 2^-9 */
    } else {
        v = ldexp((double)(8 + frac), expo - 10);  /* (1.frac) * 2^(expo-7) */
    }
    return sign ? -v : v;
}

uint8_t pkvo_f32_to_e4m3(float y)
{
    uint8_t sign = signbit(y) ? 0x80 : 0;
    if (isnan(y)) return 0x7f;
    double a = fabs((double)y);
    if (a >= 448.0) return (uint8_t)(sign | 0x7e);   /* saturate (also +-inf) */
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: value = m * 2^-9, m in [0, 8]; m == 8 is the
         * smallest normal number, whose bit pattern is 0x08 */
        double m = rint(ldexp(a, 9));
        return (uint8_t)(sign | (uint8_t)m);
    }
    int e2;
    frexp(a, &e2);
    int e = e2 - 1;                     /* a in [2^e, 2^(e+1)), e in [-6, 8] */
    double m = rint(ldexp(a, 3 - e));   /* 4-bit significand, in [8, 16] */
    if (m == 16.0) { m = 8.0; e += 1; }
    if (e > 8 || (e == 8 && m > 14.0)) return (uint8_t)(sign | 0x7e);
    return (uint8_t)(sign | (uint8_t)((e + 7) << 3) | (uint8_t)((int)m - 8));
}

static double g_e4m3[256];
static int g_e4m3_ready = 0;

static void e4m3_table_init(void)
{
    if (g_e4m3_ready) return;
    for (int i = 0; i < 256; ++i) g_e4m3[i] = pkvo_e4m3_to_f64((uint8_t)i);
    g_e4m3_ready = 1;
}

/* The code of one fp16 input under a scale: the fp16 value is exact in fp32,
 * the quotient is one correctly rounded fp32 division. */
uint8_t pkvo_quantize_e4m3(uint16_t x_f16, float scale)
{
    f16_table_init();
    volatile float x = (float)g_f16[x_f16];
    volatile float y = x / scale;
    return pkvo_f32_to_e4m3(y);
}

/* Slot-mapped append into FP8 caches (same slot rule as pkvo_append). */
int pkvo_append_f8(const uint16_t *k_new, const uint16_t *v_new, const int64_t *slot_mapping,
                   uint8_t *k_cache, uint8_t *v_cache, int num_tokens, int n_kv_heads,
                   int head_dim, int block_size, int64_t num_blocks, float k_scale,
                   float v_scale)
{
    int rc = 0;
    for (int i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= num_blocks * (int64_t)block_size) { rc = -1; continue; }
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        for (int j = 0; j < n_kv_heads; ++j) {
            const uint16_t *ksrc = k_new + ((int64_t)i * n_kv_heads + j) * head_dim;
            const uint16_t *vsrc = v_new + ((int64_t)i * n_kv_heads + j) * head_dim;
            int64_t row = ((block * n_kv_heads + j) * block_size + offset) * head_dim;
            for (int k = 0; k < head_dim; ++k) {
                k_cache[row + k] = pkvo_quantize_e4m3(ksrc[k], k_scale);
                v_cache[row + k] = pkvo_quantize_e4m3(vsrc[k], v_scale);
            }
        }
    }
    return rc;
}

/* attend_range over FP8 caches: K_t = decode(code) * k_scale and
 * V_t = decode(code) * v_scale, gathered the same way. */
static int attend_range_f8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                           double k_scale, double v_scale, const int32_t *block_tables,
                           int max_blocks_per_seq, int64_t num_blocks, double scale,
                           int n_q_heads, int n_kv_heads, int head_dim, int block_size, int b,
                           int h, int t_begin, int t_end, double *m_out, double *l_out,
                           double *acc)
{
    int group = n_q_heads / n_kv_heads;
    int j = h / group;
    int n = t_end - t_begin;
    for (int k = 0; k < head_dim; ++k) acc[k] = 0.0;
    *m_out = -INFINITY;
    *l_out = 0.0;
    if (n <= 0) return 0;
    const uint16_t *qv = q + ((int64_t)b * n_q_heads + h) * head_dim;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    if (!s) return -2;
    for (int t = t_begin; t < t_end; ++t) {
        int32_t block = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];
        if (block < 0 || block >= num_blocks) { free(s); return -1; }
        const uint8_t *kt = k_cache + (((int64_t)block * n_kv_heads + j) * block_size +
                                       t % block_size) * head_dim;
        double dot = 0.0;
        for (int k = 0; k < head_dim; ++k) dot += g_f16[qv[k]] * (g_e4m3[kt[k]] * k_scale);
        s[t - t_begin] = scale * dot;
    }
    double m = -INFINITY;
    for (int i = 0; i < n; ++i) if (s[i] > m) m = s[i];
    double l = 0.0;
    for (int i = 0; i < n; ++i) { s[i] = exp(s[i] - m); l += s[i]; }
    for (int t = t_begin; t < t_end; ++t) {
        int32_t block = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];
        const uint8_t *vt = v_cache + (((int64_t)block * n_kv_heads + j) * block_size +
                                       t % block_size) * head_dim;
        double p = s[t - t_begin];
        for (int k = 0; k < head_dim; ++k) acc[k] += p * (g_e4m3[vt[k]] * v_scale);
    }
    free(s);
    *m_out = m;
    *l_out = l;
    return 0;
}

/* pkvo_decode over FP8 caches. */
int pkvo_decode_f8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                   double k_scale, double v_scale, const int32_t *block_tables,
                   const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                   int64_t num_blocks, double scale, int n_q_heads, int n_kv_heads,
                   int head_dim, int block_size, const uint8_t *mask, double *out, double *lse,
                   int num_threads)
{
    f16_table_init();
    e4m3_table_init();
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return -1;
    for (int b = 0; b < num_seqs; ++b) {
        int L = context_lens[b];
        if (L < 0 || L > max_blocks_per_seq * block_size) return -1;
    }
    int failed = 0;
    int64_t pairs = (int64_t)num_seqs * n_q_heads;
#ifdef _OPENMP
    int nt = num_threads > 0 ? num_threads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt) reduction(| : failed)
#endif
    for (int64_t bh = 0; bh < pairs; ++bh) {
        if (mask && !mask[bh]) continue;
        int b = (int)(bh / n_q_heads);
        int h = (int)(bh % n_q_heads);
        double *acc = (double *)malloc(sizeof(double) * (size_t)head_dim);
        double m, l;
        int rc = attend_range_f8(q, k_cache, v_cache, k_scale, v_scale, block_tables,
                                 max_blocks_per_seq, num_blocks, scale, n_q_heads, n_kv_heads,
                                 head_dim, block_size, b, h, 0, context_lens[b], &m, &l, acc);
        if (rc != 0) { failed = 1; free(acc); continue; }
        for (int k = 0; k < head_dim; ++k)
            if (out) out[bh * head_dim + k] = (l > 0.0) ? acc[k] / l : 0.0;
        if (lse) lse[bh] = (l > 0.0) ? m + log(l) : -INFINITY;
        free(acc);
    }
    (void)num_threads;
    return failed ? -1 : 0;
}

/* pkvo_quantize_e4m3 over an array (n codes). */
void pkvo_quantize_e4m3_array(const uint16_t *x_f16, int64_t n, float scale, uint8_t *codes)
{
    for (int64_t i = 0; i < n; ++i) codes[i] = pkvo_quantize_e4m3(x_f16[i], scale);
}

/* pkvo_f32_to_e4m3 over an array of fp32 values. */
void pkvo_f32_to_e4m3_array(const float *y, int64_t n, uint8_t *codes)
{
    for (int64_t i = 0; i < n; ++i) codes[i] = pkvo_f32_to_e4m3(y[i]);
}

/* ---------------------------------------------------------------------------
 * Multi-token paged attention (speculative-decoding verify, chunked prefill).
 * "Roadmap: vLLM-style serving features for TornadoVM batched decode",
 * Deferred list (batch-prefill verify of draft tokens; multi-token chunked
 * prefill) and "Distributed LLM Inference Serving Platform", section 9.2
 * (chunked prefill): several new tokens of one sequence attend in one step.
 * Reading (listed in the design notes): sequence b contributes the query
 * rows [query_start[b], query_start[b+1]) of q; these n_b tokens are the last
 * n_b of its context_lens[b] = L cached tokens (already appended), so query
 * token i sits at position L - n_b + i and attends the tokens [0, L - n_b + i]
 * (causal).  q, out: [total_q][n_q_heads][head_dim]; lse: [total_q][n_q_heads].
 * ------------------------------------------------------------------------- */

/* attend_range with the query vector given directly (qv) instead of by (b, h). */
static int attend_range_qv(const uint16_t *qv, const uint16_t *k_cache, const uint16_t *v_cache,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           int64_t num_blocks, double scale, int n_q_heads, int n_kv_heads,
                           int head_dim, int block_size, int b, int h, int t_begin, int t_end,
                           double *m_out, double *l_out, double *acc)
{
    int group = n_q_heads / n_kv_heads;
    int j = h / group;
    int n = t_end - t_begin;
    for (int k = 0; k < head_dim; ++k) acc[k] = 0.0;
    *m_out = -INFINITY;
    *l_out = 0.0;
    if (n <= 0) return 0;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    if (!s) return -2;
    for (int t = t_begin; t < t_end; ++t) {
        const uint16_t *kt = token_row(k_cache, block_tables, max_blocks_per_seq, num_blocks,
                                       n_kv_heads, head_dim, block_size, b, j, t);
        if (!kt) { free(s); return -1; }
        double dot = 0.0;
        for (int k = 0; k < head_dim; ++k) dot += g_f16[qv[k]] * g_f16[kt[k]];
        s[t - t_begin] = scale * dot;
    }
    double m = -INFINITY;
    for (int i = 0; i < n; ++i) if (s[i] > m) m = s[i];
    double l = 0.0;
    for (int i = 0; i < n; ++i) { s[i] = exp(s[i] - m); l += s[i]; }
    for (int t = t_begin; t < t_end; ++t) {
        const uint16_t *vt = token_row(v_cache, block_tables, max_blocks_per_seq, num_blocks,
                                       n_kv_heads, head_dim, block_size, b, j, t);
        double p = s[t - t_begin];
        for (int k = 0; k < head_dim; ++k) acc[k] += p * g_f16[vt[k]];
    }
    free(s);
    *m_out = m;
    *l_out = l;
    return 0;
}

int pkvo_decode_multi(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                      const int32_t *block_tables, const int32_t *context_lens,
                      const int32_t *query_start, int num_seqs, int max_blocks_per_seq,
                      int64_t num_blocks, double scale, int n_q_heads, int n_kv_heads,
                      int head_dim, int block_size, double *out, double *lse, int num_threads)
{
    f16_table_init();
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return -1;
    if (query_start[0] != 0) return -1;
    for (int b = 0; b < num_seqs; ++b) {
        int L = context_lens[b];
        int nq = query_start[b + 1] - query_start[b];
        if (L < 0 || L > max_blocks_per_seq * block_size) return -1;
        if (nq < 0 || nq > L) return -1;
    }
    int total_q = query_start[num_seqs];
    int failed = 0;
    int64_t rows = (int64_t)total_q * n_q_heads;
#ifdef _OPENMP
    int nt = num_threads > 0 ? num_threads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt) reduction(| : failed)
#endif
    for (int64_t rh = 0; rh < rows; ++rh) {
        int r = (int)(rh / n_q_heads);
        int h = (int)(rh % n_q_heads);
        int b = 0;
        while (query_start[b + 1] <= r) ++b;          /* the sequence of query row r */
        int nq = query_start[b + 1] - query_start[b];
        int pos = context_lens[b] - nq + (r - query_start[b]);   /* its position */
        double *acc = (double *)malloc(sizeof(double) * (size_t)head_dim);
        double m, l;
        int rc = attend_range_qv(q + rh * head_dim, k_cache, v_cache, block_tables,
                                 max_blocks_per_seq, num_blocks, scale, n_q_heads, n_kv_heads,
                                 head_dim, block_size, b, h, 0, pos + 1, &m, &l, acc);
        if (rc != 0) { failed = 1; free(acc); continue; }
        for (int k = 0; k < head_dim; ++k)
            if (out) out[rh * head_dim + k] = (l > 0.0) ? acc[k] / l : 0.0;
        if (lse) lse[rh] = (l > 0.0) ? m + log(l) : -INFINITY;
        free(acc);
    }
    (void)num_threads;
    return failed ? -1 : 0;
}
