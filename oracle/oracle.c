/*
 * Paged decode attention: the oracle (CPU, fp64).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the paged decode path computes.  Only the test suite, the
 * smoke check and the CPU-baseline leg of the benchmark load it.  It shares no
 * code, header, table or helper with the CUDA library, and the CUDA library
 * never calls it.
 *
 * Sources (the pages describe the method; none prints the formula in full):
 *  - Block table and gather: "PagedAttention de vLLM : comment la gestion de la
 *    VRAM soutient l'inference des grands modeles" (deepsonar.com.cn), section
 *    2.2 (fixed-size blocks, a per-request table from logical to physical block
 *    numbers, the attention kernel gathers the physical blocks through it) and
 *    section 2.6 (the block table is handed to the decode kernel as a tensor).
 *  - "PagedAttention : comment optimiser la memoire GPU lors de l'inference des
 *    LLM" (deeplearn.tn), section "La table de blocs en arriere-plan" (logical
 *    block i -> physical block #n; the system reads the right tokens through
 *    the physical addresses).
 *  - GQA sharing: the deepsonar page, section 2.1 (64 attention heads share 8
 *    KV heads).  Reading taken: contiguous groups, kv_head = head / (Hq / Hkv).
 *  - Decode = one new query token that consults the stored history: "vLLM
 *    transforme la memoire GPU en systeme d'exploitation pour LLM"
 *    (chester-dev.com), section "Le cache KV est une memoire vivante".
 *  - The attention itself is softmax(q K^T * scale) V with scale passed in
 *    (1/sqrt(head_dim) in every workload).  The pages never write it out; this
 *    is the standard definition of scaled dot-product attention.
 *
 * Every function below reads fp16 inputs exactly (IEEE binary16 -> double is
 * exact) and computes in double.  The physical cache layout is an explicit
 * index function: element (block b, kv head h, offset o, dim d) of a cache sits
 * at b*stride_block + h*stride_head + o*stride_token + d (in elements), so the
 * oracle does not assume any particular layout.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* IEEE 754 binary16 -> double, written from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 *   exponent 0      : subnormal, value = fraction * 2^-24
 *   exponent 1..30  : normal,    value = (1024 + fraction) * 2^(exponent-25)
 *   exponent 31     : infinity (fraction 0) or NaN. */
double or_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -v : v;
}

/* Gather one sequence's history into contiguous double arrays
 * K[t][kv_head][d] and V[t][kv_head][d] for t in [t0, t1), walking the block
 * table: token t lives in physical block table[t / block_size] at offset
 * t % block_size. */
static void gather_sequence(double *K, double *V,
                            const uint16_t *k_cache, const uint16_t *v_cache,
                            const int32_t *table, int t0, int t1,
                            int num_kv_heads, int head_dim, int block_size,
                            int64_t stride_block, int64_t stride_head,
                            int64_t stride_token)
{
    for (int t = t0; t < t1; ++t) {
        int64_t phys = table[t / block_size];
        int64_t off = t % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t base = phys * stride_block + h * stride_head + off * stride_token;
            double *krow = K + ((int64_t)(t - t0) * num_kv_heads + h) * head_dim;
            double *vrow = V + ((int64_t)(t - t0) * num_kv_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d) {
                krow[d] = or_half_to_double(k_cache[base + d]);
                vrow[d] = or_half_to_double(v_cache[base + d]);
            }
        }
    }
}

/* Decode attention for sequences [seq_begin, seq_end).
 *
 * out      : double [num_seqs][num_heads][head_dim]
 * query    : fp16   [num_seqs][num_heads][head_dim]
 * k_cache, v_cache : fp16, addressed through the strides above
 * block_tables : int32 [num_seqs][max_blocks_per_seq]
 * context_lens : int32 [num_seqs]; L = 0 gives a zero output row.
 *
 * For each sequence i and query head h (kv head g = h / (Hq/Hkv)):
 *   s_t = scale * sum_d q[i][h][d] * K_i[t][g][d]          for t < L_i
 *   p_t = exp(s_t - max_u s_u) / sum_u exp(s_u - max_u s_u)
 *   out[i][h][d] = sum_t p_t * V_i[t][g][d]
 * Returns 0, or -1 on a bad argument or allocation failure. */
int or_paged_decode(double *out, const uint16_t *query,
                    const uint16_t *k_cache, const uint16_t *v_cache,
                    const int32_t *block_tables, const int32_t *context_lens,
                    int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                    int block_size, int max_blocks_per_seq,
                    int64_t stride_block, int64_t stride_head, int64_t stride_token,
                    double scale, int seq_begin, int seq_end)
{
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || seq_begin < 0 || seq_end > num_seqs)
        return -1;
    int group = num_heads / num_kv_heads;
    for (int i = seq_begin; i < seq_end; ++i) {
        int L = context_lens[i];
        double *orow = out + (int64_t)i * num_heads * head_dim;
        if (L <= 0) {
            memset(orow, 0, sizeof(double) * (size_t)num_heads * head_dim);
            continue;
        }
        size_t n = (size_t)L * num_kv_heads * head_dim;
        double *K = (double *)malloc(n * sizeof(double));
        double *V = (double *)malloc(n * sizeof(double));
        double *s = (double *)malloc((size_t)L * sizeof(double));
        double *q = (double *)malloc((size_t)head_dim * sizeof(double));
        if (!K || !V || !s || !q) {
            free(K); free(V); free(s); free(q);
            return -1;
        }
        gather_sequence(K, V, k_cache, v_cache,
                        block_tables + (int64_t)i * max_blocks_per_seq, 0, L,
                        num_kv_heads, head_dim, block_size,
                        stride_block, stride_head, stride_token);
        for (int h = 0; h < num_heads; ++h) {
            int g = h / group;
            const uint16_t *qh = query + ((int64_t)i * num_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d)
                q[d] = or_half_to_double(qh[d]);
            double m = -INFINITY;
            for (int t = 0; t < L; ++t) {
                const double *k = K + ((int64_t)t * num_kv_heads + g) * head_dim;
                double dot = 0.0;
                for (int d = 0; d < head_dim; ++d)
                    dot += q[d] * k[d];
                s[t] = scale * dot;
                if (s[t] > m)
                    m = s[t];
            }
            double z = 0.0;
            for (int t = 0; t < L; ++t) {
                s[t] = exp(s[t] - m);
                z += s[t];
            }
            double *o = orow + (int64_t)h * head_dim;
            for (int d = 0; d < head_dim; ++d)
                o[d] = 0.0;
            for (int t = 0; t < L; ++t) {
                double p = s[t] / z;
                const double *v = V + ((int64_t)t * num_kv_heads + g) * head_dim;
                for (int d = 0; d < head_dim; ++d)
                    o[d] += p * v[d];
            }
        }
        free(K); free(V); free(s); free(q);
    }
    return 0;
}

/* The split-context form of the same attention, in double: the context of
 * each sequence is cut into partitions of partition_tokens tokens; each
 * partition p yields its own running maximum m_p, its sum of exponentials
 * l_p = sum_t exp(s_t - m_p) and its normalised output o_p; the partitions are
 * then merged by the log-sum-exp rule
 *   M = max_p m_p,  w_p = l_p * exp(m_p - M),  out = sum_p w_p o_p / sum_p w_p.
 * This is the algebra the split-context decode and its merge step follow; in
 * exact arithmetic it equals or_paged_decode for any partition size.  The
 * incremental softmax this rests on is the one the deeplearn.tn page credits
 * to FlashAttention (section "PagedAttention vs. FlashAttention": softmax
 * computed incrementally, tile by tile). */
int or_paged_decode_split(double *out, const uint16_t *query,
                          const uint16_t *k_cache, const uint16_t *v_cache,
                          const int32_t *block_tables, const int32_t *context_lens,
                          int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                          int block_size, int max_blocks_per_seq,
                          int64_t stride_block, int64_t stride_head, int64_t stride_token,
                          double scale, int partition_tokens, int seq_begin, int seq_end)
{
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || partition_tokens <= 0 || seq_begin < 0 || seq_end > num_seqs)
        return -1;
    int group = num_heads / num_kv_heads;
    for (int i = seq_begin; i < seq_end; ++i) {
        int L = context_lens[i];
        double *orow = out + (int64_t)i * num_heads * head_dim;
        if (L <= 0) {
            memset(orow, 0, sizeof(double) * (size_t)num_heads * head_dim);
            continue;
        }
        int P = (L + partition_tokens - 1) / partition_tokens;
        size_t n = (size_t)L * num_kv_heads * head_dim;
        double *K = (double *)malloc(n * sizeof(double));
        double *V = (double *)malloc(n * sizeof(double));
        double *q = (double *)malloc((size_t)head_dim * sizeof(double));
        double *mp = (double *)malloc((size_t)P * sizeof(double));
        double *lp = (double *)malloc((size_t)P * sizeof(double));
        double *op = (double *)malloc((size_t)P * head_dim * sizeof(double));
        if (!K || !V || !q || !mp || !lp || !op) {
            free(K); free(V); free(q); free(mp); free(lp); free(op);
            return -1;
        }
        gather_sequence(K, V, k_cache, v_cache,
                        block_tables + (int64_t)i * max_blocks_per_seq, 0, L,
                        num_kv_heads, head_dim, block_size,
                        stride_block, stride_head, stride_token);
        for (int h = 0; h < num_heads; ++h) {
            int g = h / group;
            const uint16_t *qh = query + ((int64_t)i * num_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d)
                q[d] = or_half_to_double(qh[d]);
            /* partition pass */
            for (int p = 0; p < P; ++p) {
                int t0 = p * partition_tokens;
                int t1 = t0 + partition_tokens < L ? t0 + partition_tokens : L;
                double m = -INFINITY;
                for (int t = t0; t < t1; ++t) {
                    const double *k = K + ((int64_t)t * num_kv_heads + g) * head_dim;
                    double dot = 0.0;
                    for (int d = 0; d < head_dim; ++d)
                        dot += q[d] * k[d];
                    if (scale * dot > m)
                        m = scale * dot;
                }
                double l = 0.0;
                double *o = op + (int64_t)p * head_dim;
                for (int d = 0; d < head_dim; ++d)
                    o[d] = 0.0;
                for (int t = t0; t < t1; ++t) {
                    const double *k = K + ((int64_t)t * num_kv_heads + g) * head_dim;
                    const double *v = V + ((int64_t)t * num_kv_heads + g) * head_dim;
                    double dot = 0.0;
                    for (int d = 0; d < head_dim; ++d)
                        dot += q[d] * k[d];
                    double e = exp(scale * dot - m);
                    l += e;
                    for (int d = 0; d < head_dim; ++d)
                        o[d] += e * v[d];
                }
                for (int d = 0; d < head_dim; ++d)
                    o[d] /= l;
                mp[p] = m;
                lp[p] = l;
            }
            /* log-sum-exp merge */
            double M = -INFINITY;
            for (int p = 0; p < P; ++p)
                if (mp[p] > M)
                    M = mp[p];
            double wsum = 0.0;
            double *out_h = orow + (int64_t)h * head_dim;
            for (int d = 0; d < head_dim; ++d)
                out_h[d] = 0.0;
            for (int p = 0; p < P; ++p) {
                double w = lp[p] * exp(mp[p] - M);
                wsum += w;
                for (int d = 0; d < head_dim; ++d)
                    out_h[d] += w * op[(int64_t)p * head_dim + d];
            }
            for (int d = 0; d < head_dim; ++d)
                out_h[d] /= wsum;
        }
        free(K); free(V); free(q); free(mp); free(lp); free(op);
    }
    return 0;
}

/* Paged attention for several new query tokens per sequence, causal within
 * the new chunk (chunked prefill or speculative tokens over the paged cache;
 * "PagedAttention de vLLM", deepsonar.com.cn, section 2.5: a request may have
 * several tokens computed in one step -- chunked prefill, speculative
 * tokens).  Sequence i has T_i = query_start[i+1] - query_start[i] new
 * tokens, which are the last T_i of its L_i = context_lens[i] positions.
 * Query token j of sequence i (row query_start[i] + j of query and out)
 * attends to positions t <= L_i - T_i + j:
 *   s_t = scale * <q, K_t[g]>,  out = sum_t softmax(s)_t V_t[g].
 * out: double [num_query_tokens][num_heads][head_dim].  Sequences with
 * T_i = 0 have no rows.  Returns 0, or -1 on a bad argument. */
int or_paged_attention_causal(double *out, const uint16_t *query,
                              const uint16_t *k_cache, const uint16_t *v_cache,
                              const int32_t *block_tables, const int32_t *context_lens,
                              const int32_t *query_start,
                              int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                              int block_size, int max_blocks_per_seq,
                              int64_t stride_block, int64_t stride_head, int64_t stride_token,
                              double scale, int seq_begin, int seq_end)
{
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || seq_begin < 0 || seq_end > num_seqs)
        return -1;
    int group = num_heads / num_kv_heads;
    for (int i = seq_begin; i < seq_end; ++i) {
        int L = context_lens[i];
        int T = query_start[i + 1] - query_start[i];
        if (T <= 0)
            continue;
        if (T > L)
            return -1;
        size_t n = (size_t)L * num_kv_heads * head_dim;
        double *K = (double *)malloc(n * sizeof(double));
        double *V = (double *)malloc(n * sizeof(double));
        double *s = (double *)malloc((size_t)L * sizeof(double));
        double *q = (double *)malloc((size_t)head_dim * sizeof(double));
        if (!K || !V || !s || !q) {
            free(K); free(V); free(s); free(q);
            return -1;
        }
        gather_sequence(K, V, k_cache, v_cache,
                        block_tables + (int64_t)i * max_blocks_per_seq, 0, L,
                        num_kv_heads, head_dim, block_size,
                        stride_block, stride_head, stride_token);
        for (int j = 0; j < T; ++j) {
            int visible = L - T + j + 1;     /* positions 0 .. L - T + j */
            int64_t row = query_start[i] + j;
            for (int h = 0; h < num_heads; ++h) {
                int g = h / group;
                const uint16_t *qh = query + (row * num_heads + h) * head_dim;
                for (int d = 0; d < head_dim; ++d)
                    q[d] = or_half_to_double(qh[d]);
                double m = -INFINITY;
                for (int t = 0; t < visible; ++t) {
                    const double *k = K + ((int64_t)t * num_kv_heads + g) * head_dim;
                    double dot = 0.0;
                    for (int d = 0; d < head_dim; ++d)
                        dot += q[d] * k[d];
                    s[t] = scale * dot;
                    if (s[t] > m)
                        m = s[t];
                }
                double z = 0.0;
                for (int t = 0; t < visible; ++t) {
                    s[t] = exp(s[t] - m);
                    z += s[t];
                }
                double *o = out + (row * num_heads + h) * head_dim;
                for (int d = 0; d < head_dim; ++d)
                    o[d] = 0.0;
                for (int t = 0; t < visible; ++t) {
                    double p = s[t] / z;
                    const double *v = V + ((int64_t)t * num_kv_heads + g) * head_dim;
                    for (int d = 0; d < head_dim; ++d)
                        o[d] += p * v[d];
                }
            }
        }
        free(K); free(V); free(s); free(q);
    }
    return 0;
}

/* ------------------------------------------------ other cache element types
 *
 * The pages store K and V in fp16 (deepsonar page, section 2.1: two bytes per
 * element in the cache-size count).  The same attention is also computed over
 * caches of bf16 or of one-byte fp8 codes (a cache element of half the size
 * halves the bytes per token in that count).  These readers turn each stored
 * element into its exact value, from the formats' definitions. */

/* bfloat16 -> double: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
 *   exponent 0       : subnormal, fraction * 2^-133
 *   exponent 1..254  : (128 + fraction) * 2^(exponent-134)
 *   exponent 255     : infinity (fraction 0) or NaN. */
double or_bf16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 7) & 0xff;
    int frac = h & 0x7f;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -133);
    else if (expo == 255)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + frac), expo - 134);
    return sign ? -v : v;
}

/* FP8 E4M3 code -> double (the OCP 8-bit floating point E4M3 format): 1 sign
 * bit, 4 exponent bits (bias 7), 3 fraction bits; no infinities.
 *   exponent 0       : subnormal, fraction * 2^-9
 *   exponent 1..15   : (8 + fraction) * 2^(exponent-10), except
 *   exponent 15 with fraction 7: NaN.   Largest finite value 448. */
double or_e4m3_to_double(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int expo = (c >> 3) & 0xf;
    int frac = c & 0x7;
    double v;
    if (expo == 15 && frac == 7)
        v = NAN;
    else if (expo == 0)
        v = ldexp((double)frac, -9);
    else
        v = ldexp((double)(8 + frac), expo - 10);
    return sign ? -v : v;
}

enum { OR_F16 = 0, OR_BF16 = 1, OR_E4M3 = 2 };

static double elem_value(const void *base, int64_t idx, int dtype)
{
    if (dtype == OR_E4M3)
        return or_e4m3_to_double(((const uint8_t *)base)[idx]);
    if (dtype == OR_BF16)
        return or_bf16_to_double(((const uint16_t *)base)[idx]);
    return or_half_to_double(((const uint16_t *)base)[idx]);
}

/* or_paged_attention_causal over caches of element type kv_dtype (0 fp16,
 * 1 bf16, 2 fp8 E4M3) with query rows of type q_dtype (0 fp16, 1 bf16):
 * cache element e stands for value(e) * k_scale in K and value(e) * v_scale
 * in V.  query_start = NULL means one query row per sequence (the decode).
 * Strides count elements.  Returns 0, or -1 on a bad argument. */
int or_paged_attention_typed(double *out, const void *query, int q_dtype,
                             const void *k_cache, const void *v_cache, int kv_dtype,
                             double k_scale, double v_scale,
                             const int32_t *block_tables, const int32_t *context_lens,
                             const int32_t *query_start,
                             int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                             int block_size, int max_blocks_per_seq,
                             int64_t stride_block, int64_t stride_head, int64_t stride_token,
                             double scale, int seq_begin, int seq_end)
{
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || seq_begin < 0 || seq_end > num_seqs)
        return -1;
    int group = num_heads / num_kv_heads;
    for (int i = seq_begin; i < seq_end; ++i) {
        int L = context_lens[i];
        int64_t r0 = query_start ? query_start[i] : i;
        int T = query_start ? query_start[i + 1] - query_start[i] : 1;
        if (T <= 0)
            continue;
        if (L <= 0 && !query_start) {   /* decode of an empty context: zero row */
            memset(out + r0 * num_heads * head_dim, 0, sizeof(double) * (size_t)num_heads * head_dim);
            continue;
        }
        if (T > L)
            return -1;
        size_t n = (size_t)L * num_kv_heads * head_dim;
        double *K = (double *)malloc(n * sizeof(double));
        double *V = (double *)malloc(n * sizeof(double));
        double *s = (double *)malloc((size_t)L * sizeof(double));
        double *q = (double *)malloc((size_t)head_dim * sizeof(double));
        if (!K || !V || !s || !q) {
            free(K); free(V); free(s); free(q);
            return -1;
        }
        /* gather positions 0 .. L-1 through the block table, as values */
        const int32_t *table = block_tables + (int64_t)i * max_blocks_per_seq;
        for (int t = 0; t < L; ++t) {
            int64_t phys = table[t / block_size];
            int64_t off = t % block_size;
            for (int h = 0; h < num_kv_heads; ++h) {
                int64_t base = phys * stride_block + h * stride_head + off * stride_token;
                double *krow = K + ((int64_t)t * num_kv_heads + h) * head_dim;
                double *vrow = V + ((int64_t)t * num_kv_heads + h) * head_dim;
                for (int d = 0; d < head_dim; ++d) {
                    krow[d] = elem_value(k_cache, base + d, kv_dtype) * k_scale;
                    vrow[d] = elem_value(v_cache, base + d, kv_dtype) * v_scale;
                }
            }
        }
        for (int j = 0; j < T; ++j) {
            int visible = L - T + j + 1;
            int64_t row = r0 + j;
            for (int h = 0; h < num_heads; ++h) {
                int g = h / group;
                for (int d = 0; d < head_dim; ++d)
                    q[d] = elem_value(query, (row * num_heads + h) * head_dim + d, q_dtype);
                double m = -INFINITY;
                for (int t = 0; t < visible; ++t) {
                    const double *k = K + ((int64_t)t * num_kv_heads + g) * head_dim;
                    double dot = 0.0;
                    for (int d = 0; d < head_dim; ++d)
                        dot += q[d] * k[d];
                    s[t] = scale * dot;
                    if (s[t] > m)
                        m = s[t];
                }
                double z = 0.0;
                for (int t = 0; t < visible; ++t) {
                    s[t] = exp(s[t] - m);
                    z += s[t];
                }
                double *o = out + (row * num_heads + h) * head_dim;
                for (int d = 0; d < head_dim; ++d)
                    o[d] = 0.0;
                for (int t = 0; t < visible; ++t) {
                    double p = s[t] / z;
                    const double *v = V + ((int64_t)t * num_kv_heads + g) * head_dim;
                    for (int d = 0; d < head_dim; ++d)
                        o[d] += p * v[d];
                }
            }
        }
        free(K); free(V); free(s); free(q);
    }
    return 0;
}
