/*
 * pkv_oracle.c -- plain CPU oracle for attention over a block-paged KV cache.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * bench's CPU-baseline leg may load or call this library. It shares no code,
 * header, table or constant with the CUDA library; the product path never
 * links it.
 *
 * Everything here is the plain definition, written for a reader to check by
 * eye, in double precision on bf16 inputs:
 *
 *   store    -- each new token's K/V row goes to the flat cache slot named by
 *               slot_mapping (nano vllm代码详解, §2 context: the `slot_mapping`
 *               field of Context). A slot is read as block_id*block_size + offset,
 *               the flat row-major index of a [num_blocks, block_size] table (the
 *               same flat arithmetic as Mini-SGLang 源码解析（二）§6.8,
 *               `_make_2d_indices`). A negative slot is a padded token: skipped.
 *   gather   -- logical block j of a sequence lives in physical block
 *               block_table[j] (推理运行时, §分页 KV: "logical block j ->
 *               physical block b_j"); token p is row p % block_size of physical
 *               block block_table[p / block_size].
 *   attend   -- textbook softmax attention of each query row over the visible
 *               keys of its sequence, scores scaled by `scale`; query head g
 *               reads KV head g / (Hq / Hkv) (GQA: consecutive query heads share
 *               one KV head; LLM Infra 101 v0.2 summary, GQA).
 *   decode   -- one query per sequence over context_lens[i] cached tokens
 *               (nano vllm代码详解 §2 context: `context_lens`, `block_tables`).
 *   prefill  -- varlen query rows cu_seqlens_q[i]..cu_seqlens_q[i+1] over keys
 *               0..k_len-1 (cu_seqlens_k); with the causal mask, query row r of a
 *               chunk sits at absolute position (k_len - q_len) + r and sees keys
 *               0..(k_len - q_len) + r: the chunk follows its cached prefix
 *               (推理运行时 §Prefill 与 decode 输入: chunked prefill already has
 *               history in the cache; Mini-SGLang 源码解析（二）§6.6 chunks).
 *
 * Layouts (row-major, element counts):
 *   key, value        [T, Hkv, D]         bf16 bits (uint16)
 *   k_cache, v_cache  [NB, bs, Hkv, D]    bf16 bits
 *   q                 [rows, Hq, D]       bf16 bits
 *   block_tables      [S, MB]             int32
 *   out               [rows, Hq, D]       double
 *
 * Return codes: 0 ok, -1 bad argument, -2 an index (slot or block id) out of
 * range, -3 out of memory.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define PKVO_OK 0
#define PKVO_BAD_ARG (-1)
#define PKVO_OUT_OF_RANGE (-2)
#define PKVO_NO_MEMORY (-3)

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int pkvo_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void pkvo_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---------------------------------------------------------------- store -- */

int pkvo_store_kvcache(const uint16_t *key, const uint16_t *value,
                       uint16_t *k_cache, uint16_t *v_cache,
                       const int32_t *slot_mapping, int64_t num_tokens,
                       int64_t num_kv_heads, int64_t head_dim,
                       int64_t block_size, int64_t num_blocks)
{
    if (num_tokens < 0 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 || num_blocks < 1)
        return PKVO_BAD_ARG;
    const int64_t row = num_kv_heads * head_dim; /* elements of one token's K (or V) */
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue; /* padded token */
        const int64_t block_id = slot / block_size;
        const int64_t offset = slot % block_size;
        if (block_id >= num_blocks) return PKVO_OUT_OF_RANGE;
        const int64_t dst = (block_id * block_size + offset) * row;
        for (int64_t e = 0; e < row; ++e) {
            k_cache[dst + e] = key[t * row + e];
            v_cache[dst + e] = value[t * row + e];
        }
    }
    return PKVO_OK;
}

/* --------------------------------------------------------------- gather -- */

/* Copy the first n logical tokens of one sequence into contiguous [n, Hkv, D]
 * arrays, following its block table row. */
static int gather_sequence(const uint16_t *k_cache, const uint16_t *v_cache,
                           const int32_t *block_table_row, int64_t n,
                           int64_t num_kv_heads, int64_t head_dim,
                           int64_t block_size, int64_t num_blocks,
                           uint16_t *k_seq, uint16_t *v_seq)
{
    const int64_t row = num_kv_heads * head_dim;
    for (int64_t p = 0; p < n; ++p) {
        const int64_t logical_block = p / block_size;
        const int64_t offset = p % block_size;
        const int64_t physical_block = block_table_row[logical_block];
        if (physical_block < 0 || physical_block >= num_blocks) return PKVO_OUT_OF_RANGE;
        const int64_t src = (physical_block * block_size + offset) * row;
        memcpy(k_seq + p * row, k_cache + src, (size_t)row * sizeof(uint16_t));
        memcpy(v_seq + p * row, v_cache + src, (size_t)row * sizeof(uint16_t));
    }
    return PKVO_OK;
}

/* --------------------------------------------------------------- attend -- */

/* One query row of one head over keys 0..n_visible-1 of a contiguous sequence.
 * scores_buf holds at least n_visible doubles. Writes head_dim doubles to o. */
static void attend_one(const uint16_t *q_vec, const uint16_t *k_seq, const uint16_t *v_seq,
                       int64_t n_visible, int64_t kv_head, int64_t num_kv_heads,
                       int64_t head_dim, double scale, double *scores_buf, double *o)
{
    const int64_t row = num_kv_heads * head_dim;
    for (int64_t d = 0; d < head_dim; ++d) o[d] = 0.0;
    if (n_visible <= 0) return; /* nothing to attend to: zero row */

    double max_score = -INFINITY;
    for (int64_t p = 0; p < n_visible; ++p) {
        const uint16_t *k_vec = k_seq + p * row + kv_head * head_dim;
        double dot = 0.0;
        for (int64_t d = 0; d < head_dim; ++d)
            dot += bf16_bits_to_double(q_vec[d]) * bf16_bits_to_double(k_vec[d]);
        scores_buf[p] = scale * dot;
        if (scores_buf[p] > max_score) max_score = scores_buf[p];
    }
    double denom = 0.0;
    for (int64_t p = 0; p < n_visible; ++p) {
        scores_buf[p] = exp(scores_buf[p] - max_score);
        denom += scores_buf[p];
    }
    for (int64_t p = 0; p < n_visible; ++p) {
        const double weight = scores_buf[p] / denom;
        const uint16_t *v_vec = v_seq + p * row + kv_head * head_dim;
        for (int64_t d = 0; d < head_dim; ++d) o[d] += weight * bf16_bits_to_double(v_vec[d]);
    }
}

/* --------------------------------------------------------------- decode -- */

/* out[i, g, :] for every sequence i (or only those with seq_mask[i] != 0 when
 * seq_mask is not NULL; other rows are left untouched). */
int pkvo_paged_decode(double *out, const uint16_t *q,
                      const uint16_t *k_cache, const uint16_t *v_cache,
                      const int32_t *block_tables, int64_t max_blocks_per_seq,
                      const int32_t *context_lens, int64_t num_seqs,
                      int64_t num_q_heads, int64_t num_kv_heads, int64_t head_dim,
                      int64_t block_size, int64_t num_blocks, double scale,
                      const uint8_t *seq_mask)
{
    if (num_seqs < 0 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 ||
        num_blocks < 1 || max_blocks_per_seq < 0 || num_q_heads % num_kv_heads != 0)
        return PKVO_BAD_ARG;
    const int64_t group = num_q_heads / num_kv_heads;
    const int64_t row = num_kv_heads * head_dim;
    int status = PKVO_OK;
    int out_of_memory = 0;

    for (int64_t i = 0; i < num_seqs && status == PKVO_OK; ++i) {
        if (seq_mask && !seq_mask[i]) continue;
        const int64_t n = context_lens[i];
        if (n < 0 || (n + block_size - 1) / block_size > max_blocks_per_seq) return PKVO_BAD_ARG;
        uint16_t *k_seq = malloc((size_t)(n > 0 ? n : 1) * row * sizeof(uint16_t));
        uint16_t *v_seq = malloc((size_t)(n > 0 ? n : 1) * row * sizeof(uint16_t));
        if (!k_seq || !v_seq) { free(k_seq); free(v_seq); return PKVO_NO_MEMORY; }
        status = gather_sequence(k_cache, v_cache, block_tables + i * max_blocks_per_seq, n,
                                 num_kv_heads, head_dim, block_size, num_blocks, k_seq, v_seq);
        if (status == PKVO_OK) {
#pragma omp parallel for schedule(dynamic)
            for (int64_t g = 0; g < num_q_heads; ++g) {
                double *scores = malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
                if (!scores) {
#pragma omp atomic write
                    out_of_memory = 1;
                    continue;
                }
                attend_one(q + (i * num_q_heads + g) * head_dim, k_seq, v_seq, n,
                           g / group, num_kv_heads, head_dim, scale, scores,
                           out + (i * num_q_heads + g) * head_dim);
                free(scores);
            }
        }
        free(k_seq);
        free(v_seq);
    }
    return out_of_memory ? PKVO_NO_MEMORY : status;
}

/* -------------------------------------------------------------- prefill -- */

/* out[r, g, :] for every query row r (or only rows with row_mask[r] != 0). */
int pkvo_paged_prefill(double *out, const uint16_t *q,
                       const uint16_t *k_cache, const uint16_t *v_cache,
                       const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                       const int32_t *block_tables, int64_t max_blocks_per_seq,
                       int64_t num_seqs, int64_t num_q_heads, int64_t num_kv_heads,
                       int64_t head_dim, int64_t block_size, int64_t num_blocks,
                       double scale, int32_t causal, const uint8_t *row_mask)
{
    if (num_seqs < 0 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 ||
        num_blocks < 1 || max_blocks_per_seq < 0 || num_q_heads % num_kv_heads != 0)
        return PKVO_BAD_ARG;
    const int64_t group = num_q_heads / num_kv_heads;
    const int64_t row = num_kv_heads * head_dim;
    int status = PKVO_OK;
    int out_of_memory = 0;

    for (int64_t i = 0; i < num_seqs && status == PKVO_OK; ++i) {
        const int64_t q_begin = cu_seqlens_q[i];
        const int64_t q_len = cu_seqlens_q[i + 1] - q_begin;
        const int64_t k_len = cu_seqlens_k[i + 1] - cu_seqlens_k[i];
        if (q_len < 0 || k_len < 0 || (causal && q_len > k_len) ||
            (k_len + block_size - 1) / block_size > max_blocks_per_seq)
            return PKVO_BAD_ARG;
        int any = 0;
        for (int64_t r = 0; r < q_len; ++r)
            if (!row_mask || row_mask[q_begin + r]) { any = 1; break; }
        if (!any) continue;

        uint16_t *k_seq = malloc((size_t)(k_len > 0 ? k_len : 1) * row * sizeof(uint16_t));
        uint16_t *v_seq = malloc((size_t)(k_len > 0 ? k_len : 1) * row * sizeof(uint16_t));
        if (!k_seq || !v_seq) { free(k_seq); free(v_seq); return PKVO_NO_MEMORY; }
        status = gather_sequence(k_cache, v_cache, block_tables + i * max_blocks_per_seq, k_len,
                                 num_kv_heads, head_dim, block_size, num_blocks, k_seq, v_seq);
        if (status == PKVO_OK) {
            const int64_t prefix = k_len - q_len; /* cached tokens before this chunk */
#pragma omp parallel for collapse(2) schedule(dynamic)
            for (int64_t r = 0; r < q_len; ++r) {
                for (int64_t g = 0; g < num_q_heads; ++g) {
                    const int64_t qrow = q_begin + r;
                    if (row_mask && !row_mask[qrow]) continue;
                    const int64_t visible = causal ? prefix + r + 1 : k_len;
                    double *scores = malloc((size_t)(visible > 0 ? visible : 1) * sizeof(double));
                    if (!scores) {
#pragma omp atomic write
                        out_of_memory = 1;
                        continue;
                    }
                    attend_one(q + (qrow * num_q_heads + g) * head_dim, k_seq, v_seq, visible,
                               g / group, num_kv_heads, head_dim, scale, scores,
                               out + (qrow * num_q_heads + g) * head_dim);
                    free(scores);
                }
            }
        }
        free(k_seq);
        free(v_seq);
    }
    return out_of_memory ? PKVO_NO_MEMORY : status;
}

/* ------------------------------------------------------------- fp8 KV -- */
/*
 * Quantized KV cache (LLM Infra 101 v0.2, KV Quantization: the cache holds
 * low-bit values instead of bf16, at some loss of accuracy). Reading taken:
 * 8-bit OCP FP8 E4M3 codes with one fp32 scale per (token, KV head) row of
 * head_dim values, for K and V separately.
 *
 * E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0
 * holds the subnormals m * 2^-9; the code S.1111.111 is NaN and there is no
 * infinity, so the largest finite magnitude is 1.75 * 2^8 = 448.
 *
 * Quantizing a row x[0..D): amax = the largest |x_d| (NaN ignored). With
 * amax = 0 every code is 0 and the scale is 0. Otherwise, in float32 with
 * round-to-nearest-even: inv = 448 / amax, scale = amax / 448, and
 * code_d = E4M3(x_d * inv), E4M3() rounding to the nearest finite code, ties
 * to the even mantissa, magnitudes beyond 448 saturating to 448, NaN -> NaN.
 * Dequantized value: e4m3_value(code) * scale.
 */

double pkvo_e4m3_value(uint8_t code)
{
    const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Nearest finite code by exhaustive search over the 127 non-negative finite
 * codes (0x00..0x7E), ties to the code with an even mantissa. */
uint8_t pkvo_e4m3_encode(float x)
{
    if (isnan(x)) return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    int best = 0;
    double best_err = a;
    for (int c = 1; c <= 0x7E; ++c) {
        const double err = fabs(pkvo_e4m3_value((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return sign | (uint8_t)best;
}

static float bf16_bits_to_float(uint16_t bits)
{
    const uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* One row of n bf16 values -> n codes and its scale. */
void pkvo_quantize_row_fp8(const uint16_t *x, int64_t n, uint8_t *codes, float *scale)
{
    float amax = 0.0f;
    for (int64_t d = 0; d < n; ++d) {
        const float a = fabsf(bf16_bits_to_float(x[d]));
        if (a > amax) amax = a; /* NaN compares false: ignored */
    }
    if (amax == 0.0f) {
        for (int64_t d = 0; d < n; ++d) codes[d] = 0;
        *scale = 0.0f;
        return;
    }
    volatile float inv = 448.0f / amax; /* float32 division, rounded once */
    volatile float sc = amax / 448.0f;
    for (int64_t d = 0; d < n; ++d) {
        volatile float y = bf16_bits_to_float(x[d]) * inv; /* float32 product, rounded once */
        codes[d] = pkvo_e4m3_encode(y);
    }
    *scale = sc;
}

/* Store with quantization: each new token's K/V row of every KV head is
 * quantized and written to the slot named by slot_mapping (negative: skipped).
 *   k_codes, v_codes  [NB, bs, Hkv, D] uint8      k_scales, v_scales [NB*bs, Hkv] float */
int pkvo_store_kvcache_fp8(const uint16_t *key, const uint16_t *value,
                           uint8_t *k_codes, uint8_t *v_codes, float *k_scales, float *v_scales,
                           const int32_t *slot_mapping, int64_t num_tokens,
                           int64_t num_kv_heads, int64_t head_dim, int64_t block_size,
                           int64_t num_blocks)
{
    if (num_tokens < 0 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 || num_blocks < 1)
        return PKVO_BAD_ARG;
    const int64_t num_slots = num_blocks * block_size;
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) return PKVO_OUT_OF_RANGE;
        for (int64_t h = 0; h < num_kv_heads; ++h) {
            const int64_t src = (t * num_kv_heads + h) * head_dim;
            const int64_t dst = (slot * num_kv_heads + h) * head_dim;
            pkvo_quantize_row_fp8(key + src, head_dim, k_codes + dst, &k_scales[slot * num_kv_heads + h]);
            pkvo_quantize_row_fp8(value + src, head_dim, v_codes + dst, &v_scales[slot * num_kv_heads + h]);
        }
    }
    return PKVO_OK;
}

/* One query row of one head over the dequantized keys/values 0..n_visible-1
 * (double [n, Hkv, D] arrays). */
static void attend_one_dequant(const uint16_t *q_vec, const double *k_seq, const double *v_seq,
                               int64_t n_visible, int64_t kv_head, int64_t num_kv_heads,
                               int64_t head_dim, double scale, double *scores_buf, double *o)
{
    const int64_t row = num_kv_heads * head_dim;
    for (int64_t d = 0; d < head_dim; ++d) o[d] = 0.0;
    if (n_visible <= 0) return;
    double max_score = -INFINITY;
    for (int64_t p = 0; p < n_visible; ++p) {
        const double *k_vec = k_seq + p * row + kv_head * head_dim;
        double dot = 0.0;
        for (int64_t d = 0; d < head_dim; ++d) dot += bf16_bits_to_double(q_vec[d]) * k_vec[d];
        scores_buf[p] = scale * dot;
        if (scores_buf[p] > max_score) max_score = scores_buf[p];
    }
    double denom = 0.0;
    for (int64_t p = 0; p < n_visible; ++p) {
        scores_buf[p] = exp(scores_buf[p] - max_score);
        denom += scores_buf[p];
    }
    for (int64_t p = 0; p < n_visible; ++p) {
        const double weight = scores_buf[p] / denom;
        const double *v_vec = v_seq + p * row + kv_head * head_dim;
        for (int64_t d = 0; d < head_dim; ++d) o[d] += weight * v_vec[d];
    }
}

/* Decode over a quantized cache: the gathered K/V rows are dequantized
 * (code value * row scale), then the same textbook attention as
 * pkvo_paged_decode. seq_mask as there. */
int pkvo_paged_decode_fp8(double *out, const uint16_t *q,
                          const uint8_t *k_codes, const uint8_t *v_codes,
                          const float *k_scales, const float *v_scales,
                          const int32_t *block_tables, int64_t max_blocks_per_seq,
                          const int32_t *context_lens, int64_t num_seqs,
                          int64_t num_q_heads, int64_t num_kv_heads, int64_t head_dim,
                          int64_t block_size, int64_t num_blocks, double scale,
                          const uint8_t *seq_mask)
{
    if (num_seqs < 0 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 ||
        num_blocks < 1 || max_blocks_per_seq < 0 || num_q_heads % num_kv_heads != 0)
        return PKVO_BAD_ARG;
    const int64_t group = num_q_heads / num_kv_heads;
    const int64_t row = num_kv_heads * head_dim;
    int out_of_memory = 0;
    for (int64_t i = 0; i < num_seqs; ++i) {
        if (seq_mask && !seq_mask[i]) continue;
        const int64_t n = context_lens[i];
        if (n < 0 || (n + block_size - 1) / block_size > max_blocks_per_seq) return PKVO_BAD_ARG;
        double *k_seq = malloc((size_t)(n > 0 ? n : 1) * row * sizeof(double));
        double *v_seq = malloc((size_t)(n > 0 ? n : 1) * row * sizeof(double));
        if (!k_seq || !v_seq) { free(k_seq); free(v_seq); return PKVO_NO_MEMORY; }
        for (int64_t p = 0; p < n; ++p) {
            const int64_t physical_block = block_tables[i * max_blocks_per_seq + p / block_size];
            if (physical_block < 0 || physical_block >= num_blocks) {
                free(k_seq);
                free(v_seq);
                return PKVO_OUT_OF_RANGE;
            }
            const int64_t slot = physical_block * block_size + p % block_size;
            for (int64_t h = 0; h < num_kv_heads; ++h) {
                const double ks = k_scales[slot * num_kv_heads + h];
                const double vs = v_scales[slot * num_kv_heads + h];
                for (int64_t d = 0; d < head_dim; ++d) {
                    const int64_t src = (slot * num_kv_heads + h) * head_dim + d;
                    k_seq[(p * num_kv_heads + h) * head_dim + d] = pkvo_e4m3_value(k_codes[src]) * ks;
                    v_seq[(p * num_kv_heads + h) * head_dim + d] = pkvo_e4m3_value(v_codes[src]) * vs;
                }
            }
        }
#pragma omp parallel for schedule(dynamic)
        for (int64_t g = 0; g < num_q_heads; ++g) {
            double *scores = malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
            if (!scores) {
#pragma omp atomic write
                out_of_memory = 1;
                continue;
            }
            attend_one_dequant(q + (i * num_q_heads + g) * head_dim, k_seq, v_seq, n, g / group,
                               num_kv_heads, head_dim, scale, scores,
                               out + (i * num_q_heads + g) * head_dim);
            free(scores);
        }
        free(k_seq);
        free(v_seq);
    }
    return out_of_memory ? PKVO_NO_MEMORY : PKVO_OK;
}
