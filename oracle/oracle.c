/*
 * Oracle for the paged-KV hot path.  TEST INFRASTRUCTURE ONLY: the CUDA
 * library never links, includes or calls this file, and only the tests, the
 * smoke check and the benchmark's CPU-baseline leg load it.
 *
 * Plain, slow, fp32 (the precision the problem statement fixes for the
 * reference computation), written straight from the pages.  Built as usual it
 * is single-threaded.  Built with -fopenmp (only for the benchmark's all-core
 * CPU baseline) the independent rows of the work -- the gathered positions of
 * one sequence, and the (query row, head) attention rows -- are spread over
 * the host cores; each row's arithmetic and its order are the same either way,
 * so both builds give bit-identical results.
 *
 *   store   - "Inference engine: inside nano-vLLM", section "Attention in
 *             nano-vLLM" (store_kvcache): token t's K and V rows go to cache
 *             row slot_mapping[t]; a slot of -1 is skipped.
 *   gather  - "nano-vLLM Part 2: Block Tables, KV Cache, and the Path to the
 *             GPU", section 2.2: logical position j of a sequence lives in
 *             physical row block_table[j / bs] * bs + j % bs.  Paging is
 *             lossless ("How vLLM works", paged attention), so attention over
 *             the gathered rows is attention over a contiguous cache.
 *   decode  - softmax(scale * q K^T) V over the context_len gathered rows
 *             (context_len counts the token stored this step; page 1 section
 *             3.1).  Two passes: max, then exp-sum; d and j ascending.
 *   prefill - per sequence, Lq = cu_q[i+1]-cu_q[i] new queries over
 *             Lk = cu_k[i+1]-cu_k[i] keys; prefix P = Lk - Lq; query r sees
 *             keys 0..P+r (bottom-right causal; page 1 sections 2.5 and 4.1,
 *             page 4 section 8.1).  Keys j < P come from the pages, keys
 *             j >= P are this step's packed k/v rows.
 *
 * GQA: q head h reads kv head h / (H_q / H_kv) (contiguous groups).
 * Inputs are raw 16-bit words (fp16 or bf16); outputs are fp32.
 * Every function returns 0 on success and a negative code on invalid input
 * (nothing is written to the output in that case).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads of the parallel regions below, and the calling thread's index (1 and
 * 0 in the usual single-threaded build). */
static int n_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int thread_id(void)
{
#ifdef _OPENMP
    return omp_get_thread_num();
#else
    return 0;
#endif
}

#define OR_F16 0
#define OR_BF16 1

static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* IEEE 754 binary16 -> binary32, exact (every half is a float). */
static float f16_bits_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    float v;
    if (e == 0)
        v = ldexpf((float)m, -24);              /* zero or subnormal */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexpf((float)(m + 1024), e - 25);  /* 1.m * 2^(e-15) */
    return sign ? -v : v;
}

static float to_float(uint16_t h, int dtype)
{
    return dtype == OR_BF16 ? bf16_bits_to_float(h) : f16_bits_to_float(h);
}

float oracle_half_to_float(uint16_t bits, int dtype) { return to_float(bits, dtype); }

/* Threads the parallel regions use (1 in the single-threaded build). */
int oracle_num_threads(void) { return n_threads(); }

/* ---------------------------------------------------------------- store */

int oracle_store_kv(const uint16_t *k, const uint16_t *v, int64_t k_row_stride, int64_t v_row_stride,
                    uint16_t *k_cache, uint16_t *v_cache, const int32_t *slot_mapping, int32_t num_tokens,
                    int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size)
{
    const int64_t row = (int64_t)num_kv_heads * head_dim;   /* elements of one token's K (or V) */
    const int64_t rows = (int64_t)num_blocks * block_size;  /* slots in the pool */
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s < -1 || s >= rows)
            return -1;
    }
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s == -1)
            continue;
        for (int64_t e = 0; e < row; ++e) {
            k_cache[s * row + e] = k[t * k_row_stride + e];
            v_cache[s * row + e] = v[t * v_row_stride + e];
        }
    }
    return 0;
}

/* --------------------------------------------------------------- gather */

/* Physical page of logical block `logical` of a sequence's table, or -1 when
 * the table has no valid page there (past its end, -1 padding, or an id
 * outside the pool). */
static int32_t page_of(const int32_t *table, int32_t table_len, int32_t logical, int32_t num_blocks)
{
    if (logical >= table_len)
        return -1;
    int32_t page = table[logical];
    if (page < 0 || page >= num_blocks)
        return -1;
    return page;
}

/* Copies logical positions [0, n) of one sequence out of the pool into
 * dense fp32 buffers kc/vc of shape [n, H_kv, D].  Every page the context
 * needs is checked first; then the rows are copied (independent rows). */
static int gather(const uint16_t *k_cache, const uint16_t *v_cache, const int32_t *table,
                  int32_t table_len, int32_t n, int32_t num_kv_heads, int32_t head_dim,
                  int32_t num_blocks, int32_t block_size, int dtype, float *kc, float *vc)
{
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int32_t j = 0; j < n; j += block_size)
        if (page_of(table, table_len, j / block_size, num_blocks) < 0)
            return -2;
#pragma omp parallel for schedule(static)
    for (int32_t j = 0; j < n; ++j) {
        const int32_t logical = j / block_size;
        const int32_t page = page_of(table, table_len, logical, num_blocks);
        int64_t r = (int64_t)page * block_size + j % block_size;
        for (int64_t e = 0; e < row; ++e) {
            kc[j * row + e] = to_float(k_cache[r * row + e], dtype);
            vc[j * row + e] = to_float(v_cache[r * row + e], dtype);
        }
    }
    return 0;
}

/* softmax(scale * q . K_j) V over rows j in [0, n) of kv head g of the dense
 * buffers; q is one head's D values; result in out[D]. */
static void attend(const float *q, const float *kc, const float *vc, int32_t n, int32_t g,
                   int32_t num_kv_heads, int32_t head_dim, float scale, float *s, float *out)
{
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    if (n == 0) {
        for (int32_t d = 0; d < head_dim; ++d)
            out[d] = 0.0f;
        return;
    }
    float m = -INFINITY;
    for (int32_t j = 0; j < n; ++j) {
        const float *kj = kc + j * row + (int64_t)g * head_dim;
        float dot = 0.0f;
        for (int32_t d = 0; d < head_dim; ++d)
            dot += q[d] * kj[d];
        s[j] = scale * dot;
        if (s[j] > m)
            m = s[j];
    }
    float l = 0.0f;
    for (int32_t j = 0; j < n; ++j) {
        s[j] = expf(s[j] - m);
        l += s[j];
    }
    for (int32_t d = 0; d < head_dim; ++d)
        out[d] = 0.0f;
    for (int32_t j = 0; j < n; ++j) {
        const float *vj = vc + j * row + (int64_t)g * head_dim;
        for (int32_t d = 0; d < head_dim; ++d)
            out[d] += s[j] * vj[d];
    }
    for (int32_t d = 0; d < head_dim; ++d)
        out[d] /= l;
}

static int check_heads(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim)
{
    if (num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || num_q_heads % num_kv_heads)
        return -3;
    return 0;
}

/* --------------------------------------------------------------- decode */

int oracle_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                  const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                  int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                  int32_t num_blocks, int32_t block_size, float scale, int dtype, float *out)
{
    if (check_heads(num_q_heads, num_kv_heads, head_dim))
        return -3;
    const int32_t group = num_q_heads / num_kv_heads;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    int32_t max_len = 0;
    for (int32_t b = 0; b < batch; ++b) {
        if (context_lens[b] < 0)
            return -4;
        if (context_lens[b] > max_len)
            max_len = context_lens[b];
    }
    const int nt = n_threads();
    float *kc = malloc(sizeof(float) * (size_t)(max_len ? max_len : 1) * row);
    float *vc = malloc(sizeof(float) * (size_t)(max_len ? max_len : 1) * row);
    float *s = malloc(sizeof(float) * (size_t)(max_len ? max_len : 1) * nt);   /* per thread */
    float *qh = malloc(sizeof(float) * (size_t)head_dim * nt);                  /* per thread */
    float *res = malloc(sizeof(float) * (size_t)batch * num_q_heads * head_dim + 1);
    int rc = (kc && vc && s && qh && res) ? 0 : -5;
    for (int32_t b = 0; b < batch && !rc; ++b) {
        int32_t n = context_lens[b];
        rc = gather(k_cache, v_cache, block_tables + (int64_t)b * max_blocks_per_seq, max_blocks_per_seq,
                    n, num_kv_heads, head_dim, num_blocks, block_size, dtype, kc, vc);
        if (rc)
            break;
#pragma omp parallel for schedule(static)
        for (int32_t h = 0; h < num_q_heads; ++h) {
            const int t = thread_id();
            float *qt = qh + (int64_t)t * head_dim;
            const uint16_t *qb = q + ((int64_t)b * num_q_heads + h) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d)
                qt[d] = to_float(qb[d], dtype);
            attend(qt, kc, vc, n, h / group, num_kv_heads, head_dim, scale, s + (int64_t)t * (max_len ? max_len : 1),
                   res + ((int64_t)b * num_q_heads + h) * head_dim);
        }
    }
    if (!rc)
        memcpy(out, res, sizeof(float) * (size_t)batch * num_q_heads * head_dim);
    free(kc); free(vc); free(s); free(qh); free(res);
    return rc;
}

/* -------------------------------------------------------------- prefill */

int oracle_prefill_paged(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         const uint16_t *k_cache, const uint16_t *v_cache,
                         const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int32_t num_seqs,
                         const int32_t *block_tables, int32_t max_blocks_per_seq,
                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t num_blocks, int32_t block_size, float scale, int dtype, float *out)
{
    if (check_heads(num_q_heads, num_kv_heads, head_dim))
        return -3;
    const int32_t group = num_q_heads / num_kv_heads;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    const int64_t total_q = cu_seqlens_q[num_seqs];
    int32_t max_k = 0;
    for (int32_t i = 0; i < num_seqs; ++i) {
        int32_t lq = cu_seqlens_q[i + 1] - cu_seqlens_q[i];
        int32_t lk = cu_seqlens_k[i + 1] - cu_seqlens_k[i];
        if (lq < 0 || lk < lq)
            return -4;
        if (!block_tables && lk != lq)
            return -4;   /* without a block table there is no cached prefix to read */
        if (lk > max_k)
            max_k = lk;
    }
    const int nt = n_threads();
    float *kc = malloc(sizeof(float) * (size_t)(max_k ? max_k : 1) * row);
    float *vc = malloc(sizeof(float) * (size_t)(max_k ? max_k : 1) * row);
    float *s = malloc(sizeof(float) * (size_t)(max_k ? max_k : 1) * nt);   /* per thread */
    float *qh = malloc(sizeof(float) * (size_t)head_dim * nt);             /* per thread */
    float *res = malloc(sizeof(float) * (size_t)total_q * num_q_heads * head_dim + 1);
    int rc = (kc && vc && s && qh && res) ? 0 : -5;
    for (int32_t i = 0; i < num_seqs && !rc; ++i) {
        const int32_t q0 = cu_seqlens_q[i];
        const int32_t lq = cu_seqlens_q[i + 1] - q0;
        const int32_t lk = cu_seqlens_k[i + 1] - cu_seqlens_k[i];
        const int32_t prefix = lk - lq;
        if (prefix > 0)
            rc = gather(k_cache, v_cache, block_tables + (int64_t)i * max_blocks_per_seq,
                        max_blocks_per_seq, prefix, num_kv_heads, head_dim, num_blocks, block_size,
                        dtype, kc, vc);
        for (int32_t r = 0; r < lq && !rc; ++r)   /* this step's keys follow the prefix */
            for (int64_t e = 0; e < row; ++e) {
                kc[(prefix + r) * row + e] = to_float(k[(q0 + r) * row + e], dtype);
                vc[(prefix + r) * row + e] = to_float(v[(q0 + r) * row + e], dtype);
            }
        if (rc)
            break;
#pragma omp parallel for schedule(dynamic, 4)
        for (int64_t rh = 0; rh < (int64_t)lq * num_q_heads; ++rh) {   /* query row r, head h */
            const int32_t r = (int32_t)(rh / num_q_heads), h = (int32_t)(rh % num_q_heads);
            const int t = thread_id();
            float *qt = qh + (int64_t)t * head_dim;
            const uint16_t *qr = q + ((int64_t)(q0 + r) * num_q_heads + h) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d)
                qt[d] = to_float(qr[d], dtype);
            attend(qt, kc, vc, prefix + r + 1, h / group, num_kv_heads, head_dim, scale,
                   s + (int64_t)t * (max_k ? max_k : 1), res + ((int64_t)(q0 + r) * num_q_heads + h) * head_dim);
        }
    }
    if (!rc)
        memcpy(out, res, sizeof(float) * (size_t)total_q * num_q_heads * head_dim);
    free(kc); free(vc); free(s); free(qh); free(res);
    return rc;
}

/* ---------------------------------------------------------------- sample */

/* Temperature sampling as the exponential race of "From nano-vLLM to vLLM:
 * Scheduler, Paged KV Cache, Prefill/Decode, Tensor Parallelism, and
 * Sampling", section 17 (17.1, 17.4, 17.6), in fp32 and in the pages' order:
 * a_i = x_i / T; p = softmax(a) with the row maximum subtracted and the
 * denominator summed in index order; score_i = p_i / max(E_i, 1e-10); the
 * first index of the largest score.  -inf and NaN logits never win (a row
 * with no finite logit gives -1); T <= 1e-10 gives -1 (the pages' sampler
 * has no greedy path).  dtype 2 = fp32 logits, else 16-bit as to_float. */
int oracle_sample(const void *logits, int64_t row_stride, int32_t batch, int32_t vocab, int32_t dtype,
                  const float *temps, const float *noise, int32_t *tokens)
{
    if (batch < 0 || vocab <= 0 || row_stride < vocab)
        return -1;
    for (int32_t b = 0; b < batch; ++b) {
        const float t = temps[b];
        tokens[b] = -1;
        if (!(t > 1e-10f) || isinf(t))
            continue;
        float m = -INFINITY;
        for (int32_t i = 0; i < vocab; ++i) {
            const int64_t at = (int64_t)b * row_stride + i;
            const float x = dtype == 2 ? ((const float *)logits)[at] : to_float(((const uint16_t *)logits)[at], dtype);
            const float a = x / t;
            if (a > m)
                m = a;
        }
        if (!(m > -INFINITY))
            continue;
        float sum = 0.0f;
        for (int32_t i = 0; i < vocab; ++i) {
            const int64_t at = (int64_t)b * row_stride + i;
            const float x = dtype == 2 ? ((const float *)logits)[at] : to_float(((const uint16_t *)logits)[at], dtype);
            const float a = x / t;
            if (a > -INFINITY)
                sum += expf(a - m);
        }
        float best = -1.0f;
        for (int32_t i = 0; i < vocab; ++i) {
            const int64_t at = (int64_t)b * row_stride + i;
            const float x = dtype == 2 ? ((const float *)logits)[at] : to_float(((const uint16_t *)logits)[at], dtype);
            const float a = x / t;
            if (!(a > -INFINITY))
                continue;
            const float p = expf(a - m) / sum;
            const float e = noise[(int64_t)b * vocab + i];
            const float score = p / (e > 1e-10f ? e : 1e-10f);
            if (score > best) {
                best = score;
                tokens[b] = i;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------ fp8 cache */

/* OCP 8-bit floating point E4M3 ("fn": no infinities): sign, 4 exponent bits
 * with bias 7, 3 mantissa bits; exponent field 0 holds the subnormals
 * m/8 * 2^-6; S.1111.111 is NaN; the largest finite value is 448. */
static float e4m3_to_float(uint8_t b)
{
    const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
    float v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexpf((float)m, -9);
    else
        v = ldexpf((float)(m + 8), e - 10);
    return sign ? -v : v;
}

float oracle_e4m3_to_float(uint8_t b) { return e4m3_to_float(b); }

/* Nearest E4M3 code to x, ties to the even code, saturating at +-448 (the
 * fp8 KV cache's reading); NaN gives 0x7F.  Plain search over the 127
 * non-negative finite codes. */
static uint8_t float_to_e4m3(float x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const float a = fabsf(x);
    int best = 0;
    float best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const float d = fabsf(e4m3_to_float((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

uint8_t oracle_float_to_e4m3(float x) { return float_to_e4m3(x); }

/* The store into an E4M3 pool with per-tensor scales: cache = e4m3(x / scale)
 * (fp32 division, then the nearest code as above). */
int oracle_store_kv_fp8(const uint16_t *k, const uint16_t *v, int64_t k_row_stride, int64_t v_row_stride,
                        uint8_t *k_cache, uint8_t *v_cache, const int32_t *slot_mapping, int32_t num_tokens,
                        int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
                        int dtype, float k_scale, float v_scale)
{
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    const int64_t rows = (int64_t)num_blocks * block_size;
    for (int32_t t = 0; t < num_tokens; ++t)
        if (slot_mapping[t] < -1 || slot_mapping[t] >= rows)
            return -1;
    for (int32_t t = 0; t < num_tokens; ++t) {
        const int64_t s = slot_mapping[t];
        if (s == -1)
            continue;
        for (int64_t e = 0; e < row; ++e) {
            k_cache[s * row + e] = float_to_e4m3(to_float(k[t * k_row_stride + e], dtype) / k_scale);
            v_cache[s * row + e] = float_to_e4m3(to_float(v[t * v_row_stride + e], dtype) / v_scale);
        }
    }
    return 0;
}

/* Decode over an E4M3 pool: gather the context dequantized (code value *
 * scale, fp32), then the same attention as oracle_decode. */
int oracle_decode_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                      const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                      int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t num_blocks, int32_t block_size, float scale, float k_scale, float v_scale, int dtype,
                      float *out)
{
    if (check_heads(num_q_heads, num_kv_heads, head_dim))
        return -3;
    const int32_t group = num_q_heads / num_kv_heads;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    int32_t max_len = 0;
    for (int32_t b = 0; b < batch; ++b) {
        if (context_lens[b] < 0)
            return -4;
        if (context_lens[b] > max_len)
            max_len = context_lens[b];
    }
    const int nt = n_threads();
    float *kc = malloc(sizeof(float) * (size_t)(max_len ? max_len : 1) * row);
    float *vc = malloc(sizeof(float) * (size_t)(max_len ? max_len : 1) * row);
    float *s = malloc(sizeof(float) * (size_t)(max_len ? max_len : 1) * nt);   /* per thread */
    float *qh = malloc(sizeof(float) * (size_t)head_dim * nt);                  /* per thread */
    float *res = malloc(sizeof(float) * (size_t)batch * num_q_heads * head_dim + 1);
    int rc = (kc && vc && s && qh && res) ? 0 : -5;
    for (int32_t b = 0; b < batch && !rc; ++b) {
        const int32_t n = context_lens[b];
        const int32_t *table = block_tables + (int64_t)b * max_blocks_per_seq;
        for (int32_t j = 0; j < n; j += block_size)
            if (page_of(table, max_blocks_per_seq, j / block_size, num_blocks) < 0) {
                rc = -2;
                break;
            }
        if (rc)
            break;
#pragma omp parallel for schedule(static)
        for (int32_t j = 0; j < n; ++j) {
            const int32_t page = page_of(table, max_blocks_per_seq, j / block_size, num_blocks);
            const int64_t r = (int64_t)page * block_size + j % block_size;
            for (int64_t e = 0; e < row; ++e) {
                kc[j * row + e] = e4m3_to_float(k_cache[r * row + e]) * k_scale;
                vc[j * row + e] = e4m3_to_float(v_cache[r * row + e]) * v_scale;
            }
        }
#pragma omp parallel for schedule(static)
        for (int32_t h = 0; h < num_q_heads; ++h) {
            const int t = thread_id();
            float *qt = qh + (int64_t)t * head_dim;
            const uint16_t *qb = q + ((int64_t)b * num_q_heads + h) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d)
                qt[d] = to_float(qb[d], dtype);
            attend(qt, kc, vc, n, h / group, num_kv_heads, head_dim, scale, s + (int64_t)t * (max_len ? max_len : 1),
                   res + ((int64_t)b * num_q_heads + h) * head_dim);
        }
    }
    if (!rc)
        memcpy(out, res, sizeof(float) * (size_t)batch * num_q_heads * head_dim);
    free(kc); free(vc); free(s); free(qh); free(res);
    return rc;
}
