/*
 * pa_oracle.c -- reference CPU implementation of paged-KV attention.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check in
 * __graft_entry__ and the cpu_baseline leg of bench.py may load this library.
 * It shares no source, header, helper or table with the CUDA library in
 * paged_kv_continuous_gb300/csrc; neither side includes or links the other.
 *
 * Every function computes the plain definition of its operation, slowly:
 *   - all arithmetic in IEEE double (fp64); no reordering, blocking or fusion;
 *   - bf16 inputs are widened exactly (a bf16 value is the top half of an
 *     fp32 word, so the widening is a 16-bit shift, which loses nothing);
 *   - softmax is the two-pass exact form: maximum, then exp(s - max),
 *     then normalise by the sum.
 *
 * Sources (web pages this method is described on):
 *   [EAS]  koas-w, "errors and solutions" (Qwen2.5-1.5B inference from
 *          scratch), sections "KV Cache 管理" (block pool, 16-token blocks,
 *          logical->physical block_table), "自写 Triton Kernel"
 *          (store_kvcache_kernel: slot_mapping store with strides;
 *          Decode_Paged_GQAAttention_Kernel: block_table walk, online
 *          softmax, GQA head map), and "开发过程遇到的错误汇总" type 1
 *          (context_lens must include the token just stored).
 *   [MVT]  mini-vllm tutorial, "step14_7 -- Batched Forward", sections
 *          "解决方案：变长 batch（varlen）" (cu_seqlens flattening) and
 *          "cu_seqlens 只在 Attention 里才需要" (causal attention only inside
 *          a sequence; per-sequence gather_kv_from_blocks over total_len,
 *          start_positions).
 *   [CEB]  PocketLLM, "cpp_engine Batching Implementation (Phase 3.1)",
 *          section "当前 KV cache 结构" (one token row = [kv_heads, head_dim]).
 *
 * Readings where the pages are silent:
 *   - slot s of the pool is physical block s / block_size, row s % block_size;
 *   - the pool layout is [num_blocks][block_size][num_kv_heads][head_dim];
 *   - slot_mapping < 0 marks a padding token and is skipped;
 *   - context_lens[b] counts every key the sequence's last query sees,
 *     including the token stored this step ([EAS] error type 1);
 *   - a prefill chunk of q_len queries of a sequence with context_lens = n
 *     sits at positions n - q_len .. n - 1 (the paged prefix is
 *     n - q_len long, [MVT] start_positions), and query i sees keys
 *     0 .. n - q_len + i inclusive;
 *   - q head h reads kv head h / (num_q_heads / num_kv_heads);
 *   - a query with no key gets the zero vector (lse = -inf).
 *   - FP8 KV cache (codec, store and dequantisation in oracle/__init__.py):
 *     E4M3 codes with one float32 scale per kv head for K and for V, stored
 *     value = nearest-even E4M3 of x / scale (float32 division, saturated to
 *     448), read value = code value * scale; pa_oracle_decode_f64 then runs
 *     the same attention on the widened pools;
 *   - rotary embedding: rotate-half pairs (i, i + D/2), angles from
 *     caller-supplied cos / sin tables indexed [position][i], q rotated and
 *     returned, k rotated then stored (rounded once to bf16), v stored
 *     unrotated.
 *
 * Pinning: the tests check these functions against brute force over
 * contiguous K/V built before paging, closed forms (one key, equal rows,
 * zero query, two keys with known weights, head-marked and position-marked
 * values), invariance under block placement, the varlen equivalence stated
 * in [MVT], and the merge identity; the rotary embedding against the
 * complex-multiplication form, the identity at angle 0, norm preservation
 * and the relative-position property of the scores.  See
 * tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_BAD_INDEX 2
#define ORACLE_NO_MEMORY 3

/* Exact widening of a bf16 bit pattern. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t word = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

int pa_oracle_version(void) { return 1; }

int pa_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Store step ([EAS] "自写 Triton Kernel", store_kvcache_kernel): every new
 * token t with slot = slot_mapping[t] >= 0 has its K row and V row copied,
 * bit for bit, into physical block slot / block_size at row
 * slot % block_size.  Source rows are addressed through element strides so
 * that views into a fused QKV buffer work ([EAS] error type 2, second case).
 */
int pa_oracle_store_kv(const uint16_t *k, const uint16_t *v, int64_t num_tokens,
                       int64_t k_tok_stride, int64_t k_head_stride,
                       int64_t v_tok_stride, int64_t v_head_stride,
                       uint16_t *k_cache, uint16_t *v_cache, int64_t num_blocks,
                       int block_size, int num_kv_heads, int head_dim,
                       const int32_t *slot_mapping)
{
    if (num_tokens < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return ORACLE_BAD_ARG;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_blocks * block_size)
            return ORACLE_BAD_INDEX;
        int64_t block = slot / block_size;
        int64_t row = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t dst = ((block * block_size + row) * num_kv_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d) {
                k_cache[dst + d] = k[t * k_tok_stride + h * k_head_stride + d];
                v_cache[dst + d] = v[t * v_tok_stride + h * v_head_stride + d];
            }
        }
    }
    return ORACLE_OK;
}

/*
 * gather_kv_from_blocks ([MVT] "cu_seqlens 只在 Attention 里才需要"): the
 * keys of one sequence and one kv head, positions 0 .. n-1, copied out of
 * the pool into a contiguous [n][head_dim] array.  Position j lives in
 * physical block table_row[j / block_size], row j % block_size.
 */
static int gather_head(const uint16_t *cache, const int32_t *table_row, int64_t n,
                       int64_t num_blocks, int block_size, int num_kv_heads,
                       int head_dim, int kv_head, uint16_t *dst)
{
    for (int64_t j = 0; j < n; ++j) {
        int64_t block = table_row[j / block_size];
        if (block < 0 || block >= num_blocks)
            return ORACLE_BAD_INDEX;
        int64_t row = j % block_size;
        const uint16_t *src =
            cache + ((block * block_size + row) * num_kv_heads + kv_head) * head_dim;
        memcpy(dst + j * head_dim, src, (size_t)head_dim * sizeof(uint16_t));
    }
    return ORACLE_OK;
}

/*
 * Attention of one query row over keys lo .. hi-1 of contiguous K/V:
 *   s_j = scale * sum_d q[d] * K[j][d]
 *   o   = sum_j exp(s_j - m) V[j] / sum_j exp(s_j - m),  m = max_j s_j
 * Returns the natural-log sum-exp  m + ln(sum_j exp(s_j - m)), or -inf and
 * the zero vector when the range is empty.  `scores` holds hi - lo doubles.
 */
static double attend_row(const uint16_t *q, const uint16_t *K, const uint16_t *V,
                         int64_t lo, int64_t hi, int head_dim, double scale,
                         double *scores, double *o)
{
    for (int d = 0; d < head_dim; ++d)
        o[d] = 0.0;
    if (hi <= lo)
        return -INFINITY;
    double m = -INFINITY;
    for (int64_t j = lo; j < hi; ++j) {
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += bf16_to_double(q[d]) * bf16_to_double(K[j * head_dim + d]);
        double s = scale * dot;
        scores[j - lo] = s;
        if (s > m)
            m = s;
    }
    double l = 0.0;
    for (int64_t j = lo; j < hi; ++j) {
        double p = exp(scores[j - lo] - m);
        scores[j - lo] = p;
        l += p;
    }
    for (int d = 0; d < head_dim; ++d) {
        double acc = 0.0;
        for (int64_t j = lo; j < hi; ++j)
            acc += scores[j - lo] * bf16_to_double(V[j * head_dim + d]);
        o[d] = acc / l;
    }
    return m + log(l);
}

static int check_heads(int num_q_heads, int num_kv_heads)
{
    return num_q_heads > 0 && num_kv_heads > 0 && num_q_heads % num_kv_heads == 0;
}

/*
 * Varlen prefill attention over a paged cache ([MVT] "cu_seqlens 只在
 * Attention 里才需要" and "与 vLLM 的对比"): sequence s owns query rows
 * cu_seqlens[s] .. cu_seqlens[s+1]-1 of q; its keys are the first
 * context_lens[s] positions of its block_table row, gathered first and then
 * attended causally.  Query i of the chunk sits at absolute position
 * P + i with P = context_lens[s] - q_len and sees keys 0 .. P + i.
 *
 * out: [total_tokens][num_q_heads][head_dim] doubles, row-major.
 * q:   [total_tokens][num_q_heads][head_dim] bf16 bits.
 * lse: optional [total_tokens][num_q_heads] natural-log sum-exp.
 */
int pa_oracle_prefill_varlen(double *out, double *lse, const uint16_t *q,
                             const int32_t *cu_seqlens, int num_seqs,
                             const uint16_t *k_cache, const uint16_t *v_cache,
                             int64_t num_blocks, const int32_t *block_tables,
                             int64_t block_table_stride, const int32_t *context_lens,
                             int num_q_heads, int num_kv_heads, int head_dim,
                             int block_size, double scale, int num_threads)
{
    if (!check_heads(num_q_heads, num_kv_heads) || head_dim <= 0 || block_size <= 0 ||
        num_seqs < 0)
        return ORACLE_BAD_ARG;
    for (int s = 0; s < num_seqs; ++s) {
        int64_t q_len = (int64_t)cu_seqlens[s + 1] - cu_seqlens[s];
        if (q_len < 0 || context_lens[s] < q_len)
            return ORACLE_BAD_ARG;
        if ((int64_t)(context_lens[s] + block_size - 1) / block_size > block_table_stride)
            return ORACLE_BAD_ARG;
    }
    const int group = num_q_heads / num_kv_heads;
    int status = ORACLE_OK;
#ifdef _OPENMP
    if (num_threads <= 0)
        num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) collapse(2)
#endif
    for (int s = 0; s < num_seqs; ++s) {
        for (int g = 0; g < num_kv_heads; ++g) {
            const int64_t n = context_lens[s];
            const int64_t q0 = cu_seqlens[s];
            const int64_t q_len = cu_seqlens[s + 1] - q0;
            const int64_t prefix = n - q_len;
            uint16_t *K = malloc((size_t)(n > 0 ? n : 1) * head_dim * sizeof(uint16_t));
            uint16_t *V = malloc((size_t)(n > 0 ? n : 1) * head_dim * sizeof(uint16_t));
            double *scores = malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
            int rc = (K && V && scores) ? ORACLE_OK : ORACLE_NO_MEMORY;
            const int32_t *row = block_tables + (int64_t)s * block_table_stride;
            if (rc == ORACLE_OK)
                rc = gather_head(k_cache, row, n, num_blocks, block_size, num_kv_heads,
                                 head_dim, g, K);
            if (rc == ORACLE_OK)
                rc = gather_head(v_cache, row, n, num_blocks, block_size, num_kv_heads,
                                 head_dim, g, V);
            if (rc == ORACLE_OK) {
                for (int hi = 0; hi < group; ++hi) {
                    const int h = g * group + hi;
                    for (int64_t i = 0; i < q_len; ++i) {
                        const int64_t r = (q0 + i) * num_q_heads + h;
                        double e = attend_row(q + r * head_dim, K, V, 0, prefix + i + 1,
                                              head_dim, scale, scores, out + r * head_dim);
                        if (lse)
                            lse[r] = e;
                    }
                }
            }
            free(K);
            free(V);
            free(scores);
            if (rc != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
                status = rc;
            }
        }
    }
    return status;
}

/*
 * Paged GQA decode ([EAS] "自写 Triton Kernel",
 * Decode_Paged_GQAAttention_Kernel): one query row per sequence, at position
 * context_lens[b] - 1, attending every key 0 .. context_lens[b] - 1.  It is
 * the varlen prefill with q_len = 1 (same gather, same attend_row); a
 * sequence with context 0 has no key and gets the zero vector.
 *
 * out: [batch][num_q_heads][head_dim] doubles; q: [batch][num_q_heads][head_dim].
 * lse: optional [batch][num_q_heads].
 */
int pa_oracle_decode(double *out, double *lse, const uint16_t *q,
                     const uint16_t *k_cache, const uint16_t *v_cache,
                     int64_t num_blocks, const int32_t *block_tables,
                     int64_t block_table_stride, const int32_t *context_lens, int batch,
                     int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                     double scale, int num_threads)
{
    if (!check_heads(num_q_heads, num_kv_heads) || head_dim <= 0 || block_size <= 0 ||
        batch < 0)
        return ORACLE_BAD_ARG;
    for (int b = 0; b < batch; ++b)
        if (context_lens[b] < 0 ||
            (int64_t)(context_lens[b] + block_size - 1) / block_size > block_table_stride)
            return ORACLE_BAD_ARG;
    const int group = num_q_heads / num_kv_heads;
    int status = ORACLE_OK;
#ifdef _OPENMP
    if (num_threads <= 0)
        num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) collapse(2)
#endif
    for (int b = 0; b < batch; ++b) {
        for (int g = 0; g < num_kv_heads; ++g) {
            const int64_t n = context_lens[b];
            uint16_t *K = malloc((size_t)(n > 0 ? n : 1) * head_dim * sizeof(uint16_t));
            uint16_t *V = malloc((size_t)(n > 0 ? n : 1) * head_dim * sizeof(uint16_t));
            double *scores = malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
            int rc = (K && V && scores) ? ORACLE_OK : ORACLE_NO_MEMORY;
            const int32_t *row = block_tables + (int64_t)b * block_table_stride;
            if (rc == ORACLE_OK)
                rc = gather_head(k_cache, row, n, num_blocks, block_size, num_kv_heads,
                                 head_dim, g, K);
            if (rc == ORACLE_OK)
                rc = gather_head(v_cache, row, n, num_blocks, block_size, num_kv_heads,
                                 head_dim, g, V);
            if (rc == ORACLE_OK) {
                for (int hi = 0; hi < group; ++hi) {
                    const int64_t r = (int64_t)b * num_q_heads + g * group + hi;
                    double e = attend_row(q + r * head_dim, K, V, 0, n, head_dim, scale,
                                          scores, out + r * head_dim);
                    if (lse)
                        lse[r] = e;
                }
            }
            free(K);
            free(V);
            free(scores);
            if (rc != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
                status = rc;
            }
        }
    }
    return status;
}

/*
 * Attention of each sequence's decode query over one key range
 * [key_lo[b], key_hi[b]) only: the partial result of one split of a
 * flash-decoding split-K, with its natural-log sum-exp.  Used to build merge
 * inputs and to check the merge identity.
 *
 * out: [batch][num_q_heads][head_dim]; lse: [batch][num_q_heads].
 */
int pa_oracle_decode_range(double *out, double *lse, const uint16_t *q,
                           const uint16_t *k_cache, const uint16_t *v_cache,
                           int64_t num_blocks, const int32_t *block_tables,
                           int64_t block_table_stride, const int32_t *key_lo,
                           const int32_t *key_hi, int batch, int num_q_heads,
                           int num_kv_heads, int head_dim, int block_size, double scale)
{
    if (!check_heads(num_q_heads, num_kv_heads) || batch < 0)
        return ORACLE_BAD_ARG;
    const int group = num_q_heads / num_kv_heads;
    for (int b = 0; b < batch; ++b) {
        const int64_t lo = key_lo[b], hi = key_hi[b];
        if (lo < 0 || hi < lo)
            return ORACLE_BAD_ARG;
        uint16_t *K = malloc((size_t)(hi > 0 ? hi : 1) * head_dim * sizeof(uint16_t));
        uint16_t *V = malloc((size_t)(hi > 0 ? hi : 1) * head_dim * sizeof(uint16_t));
        double *scores = malloc((size_t)(hi > 0 ? hi : 1) * sizeof(double));
        int rc = (K && V && scores) ? ORACLE_OK : ORACLE_NO_MEMORY;
        const int32_t *row = block_tables + (int64_t)b * block_table_stride;
        for (int g = 0; g < num_kv_heads && rc == ORACLE_OK; ++g) {
            rc = gather_head(k_cache, row, hi, num_blocks, block_size, num_kv_heads,
                             head_dim, g, K);
            if (rc == ORACLE_OK)
                rc = gather_head(v_cache, row, hi, num_blocks, block_size, num_kv_heads,
                                 head_dim, g, V);
            for (int hi_ = 0; hi_ < group && rc == ORACLE_OK; ++hi_) {
                const int64_t r = (int64_t)b * num_q_heads + g * group + hi_;
                lse[r] = attend_row(q + r * head_dim, K, V, lo, hi, head_dim, scale, scores,
                                    out + r * head_dim);
            }
        }
        free(K);
        free(V);
        free(scores);
        if (rc != ORACLE_OK)
            return rc;
    }
    return ORACLE_OK;
}

/*
 * Log-sum-exp merge of split-K partials (flash-decoding): with partial
 * outputs o_s (each already normalised over its own keys) and their
 * natural-log sum-exps lse_s,
 *   M = max_s lse_s,  w_s = exp(lse_s - M),  o = sum_s w_s o_s / sum_s w_s.
 * Splits with lse = -inf (no keys) get weight 0; if every split is empty
 * the result is the zero vector.
 *
 * part_o: [rows][num_splits][head_dim]; part_lse: [rows][num_splits];
 * out: [rows][head_dim].
 */
void pa_oracle_merge(double *out, const double *part_o, const double *part_lse,
                     int64_t rows, int num_splits, int head_dim)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *lse = part_lse + r * num_splits;
        double M = -INFINITY;
        for (int s = 0; s < num_splits; ++s)
            if (lse[s] > M)
                M = lse[s];
        for (int d = 0; d < head_dim; ++d)
            out[r * head_dim + d] = 0.0;
        if (M == -INFINITY)
            continue;
        double wsum = 0.0;
        for (int s = 0; s < num_splits; ++s)
            wsum += lse[s] == -INFINITY ? 0.0 : exp(lse[s] - M);
        for (int d = 0; d < head_dim; ++d) {
            double acc = 0.0;
            for (int s = 0; s < num_splits; ++s) {
                if (lse[s] == -INFINITY)
                    continue;
                acc += exp(lse[s] - M) * part_o[(r * num_splits + s) * head_dim + d];
            }
            out[r * head_dim + d] = acc / wsum;
        }
    }
}

/*
 * Rotary position embedding by table lookup, rotate-half form.  [EAS]
 * "开发时间线" (days 4-5: RoPE rebuilt from the complex form into a
 * real-valued table lookup), "算子融合与模型优化" (rotate_half applied in
 * place) and "自写 Triton Kernel" (fused_rope_and_cache_store_kernel: q
 * rotated and written back contiguous, k rotated and, with v, stored
 * through slot_mapping).
 *
 * Reading: dimension i of a head pairs with dimension i + D/2 (the
 * rotate_half convention the page names), and the tables hold one angle per
 * (position, pair): for token t at p = positions[t], head h, i < D/2,
 *   c = cos_table[p * D/2 + i],  s = sin_table[p * D/2 + i],
 *   out[t][h][i]       = x[t][h][i] * c - x[t][h][i + D/2] * s
 *   out[t][h][i + D/2] = x[t][h][i + D/2] * c + x[t][h][i] * s,
 * which is x * cos + rotate_half(x) * sin with rotate_half(x) = (-x2, x1)
 * and each half-length table row repeated over both halves.  fp64; x
 * element (t, h, d) is x[t * tok_stride + h * head_dim + d]; out is
 * contiguous [num_tokens][num_heads][head_dim].
 */
int pa_oracle_rope(double *out, const uint16_t *x, int64_t num_tokens, int64_t tok_stride,
                   int num_heads, int head_dim, const int32_t *positions,
                   const float *cos_table, const float *sin_table, int64_t max_position)
{
    if (num_tokens < 0 || num_heads <= 0 || head_dim <= 0 || head_dim % 2 != 0)
        return ORACLE_BAD_ARG;
    const int half = head_dim / 2;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t p = positions[t];
        if (p < 0 || p >= max_position)
            return ORACLE_BAD_INDEX;
        for (int h = 0; h < num_heads; ++h) {
            const uint16_t *row = x + t * tok_stride + (int64_t)h * head_dim;
            double *o = out + (t * num_heads + h) * (int64_t)head_dim;
            for (int i = 0; i < half; ++i) {
                double c = (double)cos_table[p * half + i];
                double s = (double)sin_table[p * half + i];
                double x1 = bf16_to_double(row[i]);
                double x2 = bf16_to_double(row[i + half]);
                o[i] = x1 * c - x2 * s;
                o[i + half] = x2 * c + x1 * s;
            }
        }
    }
    return ORACLE_OK;
}

/*
 * Decode over pools given as fp64 values (same layout as the bf16 pools,
 * [num_blocks][block_size][num_kv_heads][head_dim]; q stays bf16).  Used
 * for the FP8 KV cache: the caller widens every stored code to its exact
 * value times its head's scale, and this is then the same gather and the
 * same two-pass softmax as pa_oracle_decode, in double.
 */
static int gather_head_f64(const double *cache, const int32_t *table_row, int64_t n,
                           int64_t num_blocks, int block_size, int num_kv_heads,
                           int head_dim, int kv_head, double *dst)
{
    for (int64_t j = 0; j < n; ++j) {
        int64_t block = table_row[j / block_size];
        if (block < 0 || block >= num_blocks)
            return ORACLE_BAD_INDEX;
        int64_t row = j % block_size;
        const double *src =
            cache + ((block * block_size + row) * num_kv_heads + kv_head) * head_dim;
        memcpy(dst + j * head_dim, src, (size_t)head_dim * sizeof(double));
    }
    return ORACLE_OK;
}

static double attend_row_f64(const uint16_t *q, const double *K, const double *V, int64_t n,
                             int head_dim, double scale, double *scores, double *o)
{
    for (int d = 0; d < head_dim; ++d)
        o[d] = 0.0;
    if (n <= 0)
        return -INFINITY;
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += bf16_to_double(q[d]) * K[j * head_dim + d];
        double s = scale * dot;
        scores[j] = s;
        if (s > m)
            m = s;
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double p = exp(scores[j] - m);
        scores[j] = p;
        l += p;
    }
    for (int d = 0; d < head_dim; ++d) {
        double acc = 0.0;
        for (int64_t j = 0; j < n; ++j)
            acc += scores[j] * V[j * head_dim + d];
        o[d] = acc / l;
    }
    return m + log(l);
}

int pa_oracle_decode_f64(double *out, double *lse, const uint16_t *q, const double *k_cache,
                         const double *v_cache, int64_t num_blocks,
                         const int32_t *block_tables, int64_t block_table_stride,
                         const int32_t *context_lens, int batch, int num_q_heads,
                         int num_kv_heads, int head_dim, int block_size, double scale)
{
    if (!check_heads(num_q_heads, num_kv_heads) || head_dim <= 0 || block_size <= 0 ||
        batch < 0)
        return ORACLE_BAD_ARG;
    for (int b = 0; b < batch; ++b)
        if (context_lens[b] < 0 ||
            (int64_t)(context_lens[b] + block_size - 1) / block_size > block_table_stride)
            return ORACLE_BAD_ARG;
    const int group = num_q_heads / num_kv_heads;
    int status = ORACLE_OK;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
#endif
    for (int b = 0; b < batch; ++b) {
        for (int g = 0; g < num_kv_heads; ++g) {
            const int64_t n = context_lens[b];
            double *K = malloc((size_t)(n > 0 ? n : 1) * head_dim * sizeof(double));
            double *V = malloc((size_t)(n > 0 ? n : 1) * head_dim * sizeof(double));
            double *scores = malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
            int rc = (K && V && scores) ? ORACLE_OK : ORACLE_NO_MEMORY;
            const int32_t *row = block_tables + (int64_t)b * block_table_stride;
            if (rc == ORACLE_OK)
                rc = gather_head_f64(k_cache, row, n, num_blocks, block_size, num_kv_heads,
                                     head_dim, g, K);
            if (rc == ORACLE_OK)
                rc = gather_head_f64(v_cache, row, n, num_blocks, block_size, num_kv_heads,
                                     head_dim, g, V);
            if (rc == ORACLE_OK) {
                for (int hi = 0; hi < group; ++hi) {
                    const int64_t r = (int64_t)b * num_q_heads + g * group + hi;
                    double e = attend_row_f64(q + r * head_dim, K, V, n, head_dim, scale,
                                              scores, out + r * head_dim);
                    if (lse)
                        lse[r] = e;
                }
            }
            free(K);
            free(V);
            free(scores);
            if (rc != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
                status = rc;
            }
        }
    }
    return status;
}
