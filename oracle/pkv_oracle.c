/*
 * pkv_oracle.c -- plain fp64 CPU oracle for one paged-attention engine step.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg may load this library.  It shares no
 * code, header, table or helper with the CUDA path, and it never calls it.
 *
 * What it computes is the plain definition, written out with no blocking, no
 * online softmax and no reordering:
 *
 *   append   -- every new token t with slot_mapping[t] >= 0 is copied, bit for
 *               bit, into physical block slot/bs at offset slot%bs of the pool.
 *               After a decode step the new token's K and V join the cache
 *               (LLM 7 - Efficient LLM Serving, sec. 3 "What the Cache
 *               Stores"); the per-token slot index is one of the fixed buffers
 *               a serving step preallocates (The Serving Playbook, "CUDA
 *               graphs and the CPU you forgot about").
 *
 *   gather   -- logical key j of request r lives in physical block
 *               block_tables[r, j / bs] at offset j % bs: the per-request
 *               block table maps logical block numbers to physical ones and
 *               attention reads through it (The Serving Playbook, "Paged KV
 *               cache"; LLM 7, sec. 3 "Paging the Cache").
 *
 *   attend   -- query i of request r (global row t = query_start_loc[r] + i)
 *               sits at position p = L_r - q_r + i and sees keys 0..p: a
 *               prefill chunk attends to what the earlier chunks wrote plus
 *               itself, causally (The Serving Playbook, "Chunked prefill").
 *               Query head h reads KV head h / g, g = Hq / Hkv (grouped-query
 *               attention shares a KV head across a group of query heads:
 *               What Actually Runs the Model, "The KV cache").  The output is
 *               softmax(scale * q K^T) V over those keys (scaled dot-product
 *               attention, LLM 7 sec. 2 "Attention Is Simple Algebra with
 *               Expensive Data Movement"), with the maximum subtracted before
 *               exponentiation (LLM 7 sec. 2 "Online Softmax Makes Tiling
 *               Possible": the subtraction prevents overflow and does not
 *               change the value).
 *
 * bf16 operands are passed as their 16-bit patterns; a bf16 value is the
 * float32 whose upper 16 bits are that pattern, widened here to double.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC (see oracle/__init__.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Thread control for the timed CPU baseline; 1 when built without OpenMP. */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Pool layout [num_blocks, Hkv, bs, D]: element (blk, h, off, d). */
static int64_t pool_index(int64_t blk, int64_t h, int64_t off, int64_t d,
                          int64_t Hkv, int64_t bs, int64_t D)
{
    return ((blk * Hkv + h) * bs + off) * D + d;
}

/*
 * Returns 0, or -1 if a slot lies beyond the pool (nothing is written then for
 * that token).
 */
int oracle_append(const uint16_t *k_new, const uint16_t *v_new,
                  const int64_t *slot_mapping, int64_t num_new_tokens,
                  int64_t Hkv, int64_t D, int64_t bs, int64_t num_blocks,
                  uint16_t *k_pool, uint16_t *v_pool)
{
    int status = 0;
    for (int64_t t = 0; t < num_new_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue; /* padding token: nothing to store */
        if (slot >= num_blocks * bs) {
            status = -1;
            continue;
        }
        int64_t blk = slot / bs;
        int64_t off = slot % bs;
        for (int64_t h = 0; h < Hkv; ++h)
            for (int64_t d = 0; d < D; ++d) {
                int64_t src = (t * Hkv + h) * D + d;
                int64_t dst = pool_index(blk, h, off, d, Hkv, bs, D);
                k_pool[dst] = k_new[src];
                v_pool[dst] = v_new[src];
            }
    }
    return status;
}

/* ------------------------------------------------------------------------
 * FP8 (e4m3) KV cache.  Eight-bit KV halves the bytes a decode step reads
 * (What Actually Runs the Model, "The KV cache"; The Serving Playbook,
 * "Quantized serving").  The format is the 8-bit float with 1 sign bit, 4
 * exponent bits (bias 7) and 3 mantissa bits, no infinities, one NaN pattern
 * per sign (exponent and mantissa all ones), largest finite magnitude 448.
 * [READING] A stored code is round-to-nearest-even of x / scale computed in
 * fp32, saturated to +-448; the value it stands for is decode(code) * scale.
 * ------------------------------------------------------------------------ */

double oracle_e4m3_decode(uint8_t c)
{
    const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);               /* subnormal: m/8 * 2^(1-7) */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Nearest finite code by exhaustive search; ties go to the even code. */
uint8_t oracle_e4m3_encode(float x)
{
    if (x != x)
        return 0x7F;
    const double a = fabs((double)x);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {           /* non-negative finite codes */
        const double err = fabs(oracle_e4m3_decode((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best_err = err;
            best = c;
        }
    }
    if (a >= 448.0)
        best = 0x7E;                            /* saturate */
    return (uint8_t)(signbit(x) ? (best | 0x80) : best);  /* -0 keeps its sign */
}

static float bf16_bits_to_float(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * Append into fp8 pools: code = encode(fp32(x) / fp32(scale[h])).
 * k_scale / v_scale: [Hkv] floats.  Returns -1 if a slot lies beyond the pool.
 */
int oracle_append_fp8(const uint16_t *k_new, const uint16_t *v_new,
                      const int64_t *slot_mapping, int64_t num_new_tokens, int64_t Hkv,
                      int64_t D, int64_t bs, int64_t num_blocks, const float *k_scale,
                      const float *v_scale, uint8_t *k_pool, uint8_t *v_pool)
{
    int status = 0;
    for (int64_t t = 0; t < num_new_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_blocks * bs) {
            status = -1;
            continue;
        }
        const int64_t blk = slot / bs, off = slot % bs;
        for (int64_t h = 0; h < Hkv; ++h)
            for (int64_t d = 0; d < D; ++d) {
                const int64_t src = (t * Hkv + h) * D + d;
                const int64_t dst = pool_index(blk, h, off, d, Hkv, bs, D);
                const float kq = bf16_bits_to_float(k_new[src]) / k_scale[h];
                const float vq = bf16_bits_to_float(v_new[src]) / v_scale[h];
                k_pool[dst] = oracle_e4m3_encode(kq);
                v_pool[dst] = oracle_e4m3_encode(vq);
            }
    }
    return status;
}

/*
 * Whole-block copy between pools of layout [blocks, Hkv, bs, D]: for each
 * pair i, block pairs[2i] of the source pools goes to block pairs[2i+1] of the
 * destination pools (copy-on-write of a shared block; swapping blocks out to
 * CPU memory and back: LLM 7 - Efficient LLM Serving, sec. 3 "Sharing and
 * Preemption").  Returns -1 (copying nothing for that pair) if a block lies
 * outside its pool.
 */
int oracle_copy_blocks(const uint16_t *k_src, const uint16_t *v_src, uint16_t *k_dst,
                       uint16_t *v_dst, const int64_t *pairs, int64_t num_pairs,
                       int64_t src_blocks, int64_t dst_blocks, int64_t Hkv, int64_t bs,
                       int64_t D)
{
    int status = 0;
    const int64_t per_block = Hkv * bs * D;
    for (int64_t i = 0; i < num_pairs; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
            status = -1;
            continue;
        }
        for (int64_t e = 0; e < per_block; ++e) {
            k_dst[dst * per_block + e] = k_src[src * per_block + e];
            v_dst[dst * per_block + e] = v_src[src * per_block + e];
        }
    }
    return status;
}

/*
 * q        [Tq, Hq, D]   bf16 bits, Tq = query_start_loc[R]
 * k_pool   [num_blocks, Hkv, bs, D] bf16 bits (v_pool the same)
 * block_tables [R, max_blocks] int32; seq_lens [R] int32 (L_r, this step's
 *          tokens included); query_start_loc [R+1] int32
 * out      [Tq, Hq, D]   fp64
 *
 * Returns 0, -1 for inconsistent arguments (q_r > L_r, a table entry outside
 * the pool, L_r beyond the table), -2 if memory for a score row is exhausted.
 */
static int paged_attention_impl(const uint16_t *q, const uint16_t *k_pool,
                                const uint16_t *v_pool, const uint8_t *k8, const uint8_t *v8,
                                const float *k_scale, const float *v_scale,
                                const int32_t *block_tables,
                                const int32_t *seq_lens,
                                const int32_t *query_start_loc, int32_t R,
                                int32_t Hq, int32_t Hkv, int32_t D, int32_t bs,
                                int32_t num_blocks, int32_t max_blocks, double scale,
                                double *out)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || bs <= 0)
        return -1;
    const int32_t g = Hq / Hkv;
    for (int32_t r = 0; r < R; ++r) {
        int32_t q_r = query_start_loc[r + 1] - query_start_loc[r];
        int32_t L = seq_lens[r];
        if (q_r < 0 || q_r > L || L > max_blocks * bs)
            return -1;
        for (int32_t j = 0; j < L; ++j) {
            int32_t blk = block_tables[(int64_t)r * max_blocks + j / bs];
            if (blk < 0 || blk >= num_blocks)
                return -1;
        }
    }
    const int32_t Tq = query_start_loc[R];
    int status = 0;

    /* One independent row per (query token, query head). */
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t row = 0; row < (int64_t)Tq * Hq; ++row) {
        const int32_t t = (int32_t)(row / Hq);
        const int32_t h = (int32_t)(row % Hq);
        int32_t r = 0;
        while (query_start_loc[r + 1] <= t)
            ++r;
        const int32_t q_r = query_start_loc[r + 1] - query_start_loc[r];
        const int32_t i = t - query_start_loc[r];
        const int32_t L = seq_lens[r];
        const int32_t p = L - q_r + i; /* this query's own position */
        const int32_t kh = h / g;
        double *o = out + ((int64_t)t * Hq + h) * D;

        double *s = (double *)malloc(sizeof(double) * (size_t)(p + 1));
        if (s == NULL) {
            #pragma omp atomic write
            status = -2;
            continue;
        }
        /* s_j = scale * <q[t,h,:], K_r[j,kh,:]> for j = 0..p */
        double m = -INFINITY;
        for (int32_t j = 0; j <= p; ++j) {
            int32_t blk = block_tables[(int64_t)r * max_blocks + j / bs];
            int32_t off = j % bs;
            double dot = 0.0;
            for (int32_t d = 0; d < D; ++d) {
                const int64_t e = pool_index(blk, kh, off, d, Hkv, bs, D);
                const double kv = k8 ? oracle_e4m3_decode(k8[e]) * (double)k_scale[kh]
                                     : bf16_bits_to_double(k_pool[e]);
                dot += bf16_bits_to_double(q[((int64_t)t * Hq + h) * D + d]) * kv;
            }
            s[j] = scale * dot;
            if (s[j] > m)
                m = s[j];
        }
        /* softmax weights with the maximum subtracted, then the weighted sum */
        double z = 0.0;
        for (int32_t j = 0; j <= p; ++j) {
            s[j] = exp(s[j] - m);
            z += s[j];
        }
        for (int32_t d = 0; d < D; ++d)
            o[d] = 0.0;
        for (int32_t j = 0; j <= p; ++j) {
            int32_t blk = block_tables[(int64_t)r * max_blocks + j / bs];
            int32_t off = j % bs;
            double w = s[j] / z;
            for (int32_t d = 0; d < D; ++d) {
                const int64_t e = pool_index(blk, kh, off, d, Hkv, bs, D);
                const double vv = v8 ? oracle_e4m3_decode(v8[e]) * (double)v_scale[kh]
                                     : bf16_bits_to_double(v_pool[e]);
                o[d] += w * vv;
            }
        }
        free(s);
    }
    return status;
}

int oracle_paged_attention(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                           const int32_t *block_tables, const int32_t *seq_lens,
                           const int32_t *query_start_loc, int32_t R, int32_t Hq,
                           int32_t Hkv, int32_t D, int32_t bs, int32_t num_blocks,
                           int32_t max_blocks, double scale, double *out)
{
    return paged_attention_impl(q, k_pool, v_pool, NULL, NULL, NULL, NULL, block_tables,
                                seq_lens, query_start_loc, R, Hq, Hkv, D, bs, num_blocks,
                                max_blocks, scale, out);
}

/* The same attention over fp8 pools: K = decode(code) * k_scale[h], V alike. */
int oracle_paged_attention_fp8(const uint16_t *q, const uint8_t *k_pool, const uint8_t *v_pool,
                               const float *k_scale, const float *v_scale,
                               const int32_t *block_tables, const int32_t *seq_lens,
                               const int32_t *query_start_loc, int32_t R, int32_t Hq,
                               int32_t Hkv, int32_t D, int32_t bs, int32_t num_blocks,
                               int32_t max_blocks, double scale, double *out)
{
    return paged_attention_impl(q, NULL, NULL, k_pool, v_pool, k_scale, v_scale, block_tables,
                                seq_lens, query_start_loc, R, Hq, Hkv, D, bs, num_blocks,
                                max_blocks, scale, out);
}
