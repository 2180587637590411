/*
 * oracle.c -- plain, slow, fp64 CPU definition of the paged KV-cache decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the CPU
 * baseline leg of bench.py may load or call this file.  It shares no code,
 * header, table or helper with the CUDA library; the product never links it.
 *
 * What it follows (page / section of the source pages):
 *   - "vLLM의 핵심 원리 PagedAttention 파헤치기" (donmain.dev), section
 *     "KV Cache를 블록으로 쪼개다": fixed 16-token blocks, a per-sequence block
 *     table that maps logical block i to a physical block, and a gather step
 *     after which attention behaves exactly as on contiguous K/V.
 *   - same page, section "낭비가 4% 밑으로": only the last block of a sequence
 *     holds empty slots (100 tokens -> 7 blocks, 12 empty slots).
 *   - "LLM 추론 배칭 전략 정리" (velog.io), section 5 "왜 이게 가능한가":
 *     a physical block is a block number inside one pool reserved up front.
 *   - "vLLM-and-PagedAttention-KR" (ghkdgus29.github.io), section
 *     "KV Cache Size 계산 방법": bytes per token = 2 x H x L x B.
 *   - "kv-cache-by-model" (sotaaz.com), section 1 "Full attention":
 *     per layer, per token, 2 (K and V) x kv_heads x head_dim x 2 bytes.
 *
 * Readings where the pages are silent:
 *   R1  pool layout [num_blocks][num_kv_heads][block_size][head_dim];
 *   R2  slot = physical_block * block_size + offset, negative slot = skip;
 *   R3  query head h reads kv head h / (num_q_heads / num_kv_heads);
 *   R7  a sequence with context length 0 yields an all-zero output row.
 *
 * Parity of every function below is pinned in tests/test_oracle_pins.py by
 * values the pages print, closed forms, invariants and brute force.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- numbers */

/* IEEE-754 binary16 bit pattern -> exact double. */
double oracle_f16_to_double(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);              /* subnormal: frac * 2^-24 */
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), expo - 25); /* (1.frac) * 2^(e-15) */
    return sign ? -mag : mag;
}

/* bfloat16 bit pattern (upper half of a binary32) -> exact double. */
double oracle_bf16_to_double(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 7) & 0xff;
    int frac = bits & 0x7f;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -133);             /* subnormal: frac * 2^-133 */
    else if (expo == 255)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(128 + frac), expo - 134); /* (1.frac) * 2^(e-127) */
    return sign ? -mag : mag;
}

static double to_double(uint16_t bits, int is_bf16)
{
    return is_bf16 ? oracle_bf16_to_double(bits) : oracle_f16_to_double(bits);
}

/* ---------------------------------------------------------------- sizing */

/* Bytes of KV cache one token occupies: 2 (K and V) x kv_heads x head_dim x
 * elem_bytes per layer, times the number of layers ("KV Cache Size 계산 방법";
 * "kv-cache-by-model" section 1).  For MHA, kv_heads x head_dim is the hidden
 * size H of the formula 2 x H x L x B. */
int64_t oracle_kv_bytes_per_token(int32_t layers, int32_t kv_heads,
                                  int32_t head_dim, int32_t elem_bytes)
{
    return (int64_t)2 * kv_heads * head_dim * elem_bytes * layers;
}

/* Blocks a sequence of n tokens owns when blocks are handed out one at a time
 * as the sequence grows: the first token opens block 0, token 17 (of a 16-token
 * block) opens block 1 ("KV Cache를 블록으로 쪼개다"). */
int64_t oracle_blocks_for_tokens(int64_t n, int32_t block_size)
{
    int64_t blocks = 0;
    for (int64_t tok = 0; tok < n; ++tok)
        if (tok % block_size == 0)   /* this token finds every slot taken */
            ++blocks;
    return blocks;
}

/* Empty slots left in a sequence's blocks ("낭비가 4% 밑으로"). */
int64_t oracle_empty_slots(int64_t n, int32_t block_size)
{
    return oracle_blocks_for_tokens(n, block_size) * block_size - n;
}

/* ------------------------------------------------------------- cache write */

/* Store each new token's K and V rows into its slot (R1, R2).  Rows are copied
 * as bit patterns, never converted.  Returns the number of tokens whose slot
 * lies beyond the pool (those are skipped, as are negative slots). */
int64_t oracle_cache_write(const uint16_t *k_new, const uint16_t *v_new,
                           const int64_t *slot_mapping, int64_t num_tokens,
                           int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, int64_t num_blocks,
                           uint16_t *k_pool, uint16_t *v_pool)
{
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_blocks * block_size) {
            ++bad;
            continue;
        }
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        for (int32_t g = 0; g < num_kv_heads; ++g) {
            for (int32_t d = 0; d < head_dim; ++d) {
                int64_t src = (t * num_kv_heads + g) * head_dim + d;
                int64_t dst = ((block * num_kv_heads + g) * block_size + offset) * head_dim + d;
                k_pool[dst] = k_new[src];
                v_pool[dst] = v_new[src];
            }
        }
    }
    return bad;
}

/* Copy-on-write: block dst_ids[i] becomes a copy of block src_ids[i], K and V,
 * every kv head and slot ("vLLM-and-PagedAttention-KR", "Parallel Sampling
 * decoding": a shared block that one sample writes into is copied first).
 * Pairs are applied in order.  Returns the number of pairs naming a block
 * outside the pool (those are skipped). */
int64_t oracle_block_copy(uint16_t *k_pool, uint16_t *v_pool, const int32_t *src_ids,
                          const int32_t *dst_ids, int64_t n, int32_t num_kv_heads,
                          int32_t block_size, int32_t head_dim, int64_t num_blocks)
{
    int64_t bad = 0;
    int64_t per_block = (int64_t)num_kv_heads * block_size * head_dim;
    for (int64_t i = 0; i < n; ++i) {
        int64_t src = src_ids[i], dst = dst_ids[i];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            ++bad;
            continue;
        }
        for (int64_t e = 0; e < per_block; ++e) {
            k_pool[dst * per_block + e] = k_pool[src * per_block + e];
            v_pool[dst * per_block + e] = v_pool[src * per_block + e];
        }
    }
    return bad;
}

/* ------------------------------------------------------------ 8-bit KV cache */

/* fp32 value -> IEEE binary16 bits, round to nearest, ties to even (finite,
 * non-negative inputs below 65520).  Written from the format's definition. */
uint16_t oracle_f32_to_f16_bits(float f)
{
    double a = fabs((double)f);
    uint16_t sign = f < 0 ? 0x8000 : 0;
    if (a == 0.0) return sign;
    if (a < ldexp(1.0, -14))                       /* subnormal: units of 2^-24 */
        return sign | (uint16_t)rint(a / ldexp(1.0, -24));
    int e;
    double m = frexp(a, &e);                       /* a = m * 2^e, m in [0.5, 1) */
    double q = rint((2.0 * m - 1.0) * 1024.0);     /* 10 fraction bits of 1.f * 2^(e-1) */
    int ex = e - 1 + 15;
    if (q == 1024.0) { q = 0.0; ++ex; }
    return sign | (uint16_t)(ex << 10) | (uint16_t)q;
}

/* 8-bit quantisation of groups of 32 values with one fp16 scale per group
 * ("kv-cache-by-model", section 1: an 8-bit cache stores a separate scale for
 * every group of 32 values, 53.1 % of the fp16 size).  Reading of the rule:
 * amax = max |x|, d = fp16(min(amax / 127, 65504)), code = clamp(rint(x / d),
 * -127, 127) in fp32 (codes 0 when d = 0); the value the cache holds is
 * code * d. */
void oracle_quantize_q8(const uint16_t *x, int64_t num_groups, int is_bf16, int8_t *codes,
                        uint16_t *scales)
{
    for (int64_t gi = 0; gi < num_groups; ++gi) {
        const uint16_t *xs = x + gi * 32;
        float amax = 0.0f;
        for (int i = 0; i < 32; ++i) {
            float v = (float)to_double(xs[i], is_bf16);
            if (fabsf(v) > amax) amax = fabsf(v);
        }
        float d32 = amax / 127.0f;
        if (d32 > 65504.0f) d32 = 65504.0f;
        uint16_t h = oracle_f32_to_f16_bits(d32);
        float dq = (float)oracle_f16_to_double(h);
        scales[gi] = h;
        for (int i = 0; i < 32; ++i) {
            float v = (float)to_double(xs[i], is_bf16);
            int c = 0;
            if (dq != 0.0f) {
                float r = rintf(v / dq);
                c = r > 127.0f ? 127 : (r < -127.0f ? -127 : (int)r);
            }
            codes[gi * 32 + i] = (int8_t)c;
        }
    }
}

/* Bytes per token of an 8-bit cache: 2 (K, V) x kv_heads x layers x
 * (head_dim one-byte codes + head_dim / 32 two-byte scales). */
int64_t oracle_q8_bytes_per_token(int32_t layers, int32_t kv_heads, int32_t head_dim)
{
    return (int64_t)kv_heads * 2 * layers * (head_dim + head_dim / 32 * 2);
}

/* Cache write into an 8-bit pool.  Layouts (per (block, kv head) slab):
 *   k_codes [num_blocks][Hkv][block_size][head_dim]   (token rows)
 *   v_codes [num_blocks][Hkv][head_dim][block_size]   (dimension rows)
 *   k_scales, v_scales [num_blocks][Hkv][block_size][head_dim / 32]
 * Slots as in oracle_cache_write.  Returns the number of out-of-pool slots. */
int64_t oracle_cache_write_q8(const uint16_t *k_new, const uint16_t *v_new,
                              const int64_t *slot_mapping, int64_t num_tokens,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              int64_t num_blocks, int is_bf16, int8_t *k_codes, int8_t *v_codes,
                              uint16_t *k_scales, uint16_t *v_scales)
{
    int64_t bad = 0;
    int32_t ng = head_dim / 32;
    int8_t *kc = (int8_t *)malloc((size_t)head_dim);
    int8_t *vc = (int8_t *)malloc((size_t)head_dim);
    uint16_t *ks = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)ng);
    uint16_t *vs = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)ng);
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * block_size) { ++bad; continue; }
        int64_t block = slot / block_size, offset = slot % block_size;
        for (int32_t g = 0; g < num_kv_heads; ++g) {
            int64_t src = (t * num_kv_heads + g) * head_dim;
            oracle_quantize_q8(k_new + src, ng, is_bf16, kc, ks);
            oracle_quantize_q8(v_new + src, ng, is_bf16, vc, vs);
            int64_t slab = block * num_kv_heads + g;
            for (int32_t d = 0; d < head_dim; ++d) {
                k_codes[(slab * block_size + offset) * head_dim + d] = kc[d];
                v_codes[(slab * head_dim + d) * block_size + offset] = vc[d];
            }
            for (int32_t i = 0; i < ng; ++i) {
                k_scales[(slab * block_size + offset) * ng + i] = ks[i];
                v_scales[(slab * block_size + offset) * ng + i] = vs[i];
            }
        }
    }
    free(kc); free(vc); free(ks); free(vs);
    return bad;
}

/* ---------------------------------------------------------- attention core */

/* Softmax attention of one query over n contiguous rows, by the definition:
 *   x_j = scale * <q, k_j>,  w_j = exp(x_j - max x),  o = sum_j w_j v_j / sum_j w_j.
 * Also returns the unnormalised accumulator pieces (max, sum of weights) when
 * asked, which is what a split of the rows hands to a merge. */
static void attend_rows(const double *q, const double *K, const double *V,
                        int64_t n, int32_t D, double scale, double *x,
                        double *out, double *acc_out, double *m_out, double *l_out)
{
    if (n == 0) {
        for (int32_t d = 0; d < D; ++d) out[d] = 0.0;
        if (acc_out) for (int32_t d = 0; d < D; ++d) acc_out[d] = 0.0;
        if (m_out) *m_out = -INFINITY;
        if (l_out) *l_out = 0.0;
        return;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d)
            dot += q[d] * K[j * D + d];
        x[j] = scale * dot;
        if (x[j] > m) m = x[j];
    }
    double Z = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        x[j] = exp(x[j] - m);
        Z += x[j];
    }
    for (int32_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t j = 0; j < n; ++j)
            acc += x[j] * V[j * D + d];
        if (acc_out) acc_out[d] = acc;
        out[d] = acc / Z;
    }
    if (m_out) *m_out = m;
    if (l_out) *l_out = Z;
}

/* Plain single-query attention on contiguous fp64 arrays: q[D], K[n][D],
 * V[n][D] -> out[D].  The result the paged gather must reproduce. */
void oracle_dense_attention(const double *q, const double *K, const double *V,
                            int64_t n, int32_t head_dim, double scale, double *out)
{
    double *x = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    attend_rows(q, K, V, n, head_dim, scale, x, out, NULL, NULL, NULL);
    free(x);
}

/* Rebuild a sequence's contiguous K/V for kv head g from its block table:
 * logical token j lives in block_table[j / block_size] at row j % block_size.
 * Returns 0, or -1 when a table entry is not a block of the pool. */
static int gather_sequence(const uint16_t *k_pool, const uint16_t *v_pool,
                           const int32_t *table_row, int64_t n, int32_t g,
                           int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, int64_t num_blocks, int is_bf16,
                           double *K, double *V)
{
    for (int64_t j = 0; j < n; ++j) {
        int64_t block = table_row[j / block_size];
        int64_t offset = j % block_size;
        if (block < 0 || block >= num_blocks)
            return -1;
        int64_t base = ((block * num_kv_heads + g) * block_size + offset) * head_dim;
        for (int32_t d = 0; d < head_dim; ++d) {
            K[j * head_dim + d] = to_double(k_pool[base + d], is_bf16);
            V[j * head_dim + d] = to_double(v_pool[base + d], is_bf16);
        }
    }
    return 0;
}

/* PagedAttention decode by definition: for every sequence s and query head h,
 * gather the sequence's K/V through its block table and run plain softmax
 * attention of q[s][h] over its context_lens[s] tokens, in fp64.
 *   q        [num_seqs][num_q_heads][head_dim]   fp16/bf16 bits
 *   k_pool   [num_blocks][num_kv_heads][block_size][head_dim] (R1), same v_pool
 *   tables   [num_seqs][max_blocks_per_seq] int32
 *   out      [num_seqs][num_q_heads][head_dim]   fp64
 * A sequence whose length exceeds its table, is negative, or whose table names
 * a block outside the pool gets a zero row and counts in the return value.
 * num_threads > 1 spreads independent (sequence, head) rows over threads;
 * the result does not depend on it. */
int64_t oracle_paged_decode(const uint16_t *q, const uint16_t *k_pool,
                            const uint16_t *v_pool, const int32_t *block_tables,
                            int32_t max_blocks_per_seq, const int32_t *context_lens,
                            int32_t num_seqs, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int64_t num_blocks, int is_bf16,
                            double scale, double *out, int num_threads)
{
    int32_t group = num_q_heads / num_kv_heads;  /* query heads per kv head (R3) */
    int64_t bad = 0;
    int64_t rows = (int64_t)num_seqs * num_q_heads;
#ifdef _OPENMP
    if (num_threads < 1) num_threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(+ : bad)
#endif
    for (int64_t r = 0; r < rows; ++r) {
        int32_t s = (int32_t)(r / num_q_heads);
        int32_t h = (int32_t)(r % num_q_heads);
        int32_t g = h / group;
        int64_t n = context_lens[s];
        double *o = out + r * head_dim;
        if (n < 0 || n > (int64_t)max_blocks_per_seq * block_size) {
            for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
            if (h == 0) ++bad;
            continue;
        }
        double *K = (double *)malloc(sizeof(double) * (size_t)(n * head_dim + 1));
        double *V = (double *)malloc(sizeof(double) * (size_t)(n * head_dim + 1));
        double *x = (double *)malloc(sizeof(double) * (size_t)(n + 1));
        double *qv = (double *)malloc(sizeof(double) * (size_t)head_dim);
        const int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
        if (gather_sequence(k_pool, v_pool, row, n, g, num_kv_heads, head_dim,
                            block_size, num_blocks, is_bf16, K, V) != 0) {
            for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
            if (h == 0) ++bad;
        } else {
            for (int32_t d = 0; d < head_dim; ++d)
                qv[d] = to_double(q[r * head_dim + d], is_bf16);
            attend_rows(qv, K, V, n, head_dim, scale, x, o, NULL, NULL, NULL);
        }
        free(K); free(V); free(x); free(qv);
    }
    return bad;
}

/* Chunked prefill by definition ("vLLM과 Ollama의 차이", chunked prefill: a long
 * prompt is cut into chunks that join the decode batch; "LLM 추론 배칭 전략
 * 정리" section 0: a prefill step processes the prompt's tokens together).
 * Sequence s holds context_lens[s] tokens in the cache, the last C_s of which
 * (C_s = query_start[s+1] - query_start[s]) are this chunk; its query row
 * r = query_start[s] + j sits at position p = context_lens[s] - C_s + j and
 * attends, as in any causal decoder, to the sequence's tokens 0..p, gathered
 * through the block table.
 *   q, out  [num_tokens][num_q_heads][head_dim] (out in fp64)
 * Rows of a sequence with a bad length, chunk or table entry are zero and
 * counted once per sequence in the return value. */
int64_t oracle_paged_prefill(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                             const int32_t *block_tables, int32_t max_blocks_per_seq,
                             const int32_t *query_start, const int32_t *context_lens,
                             int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                             int32_t head_dim, int32_t block_size, int64_t num_blocks,
                             int is_bf16, double scale, double *out, int num_threads)
{
    int32_t group = num_q_heads / num_kv_heads;
    int64_t bad = 0;
#ifdef _OPENMP
    if (num_threads < 1) num_threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(+ : bad)
#endif
    for (int32_t s = 0; s < num_seqs; ++s) {
        int64_t r0 = query_start[s], r1 = query_start[s + 1];
        int64_t C = r1 - r0, L = context_lens[s];
        int ok = C >= 0 && L >= C && L <= (int64_t)max_blocks_per_seq * block_size;
        double *K = NULL, *V = NULL, *x = NULL, *qv = NULL;
        const int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
        if (ok && C > 0) {
            K = (double *)malloc(sizeof(double) * (size_t)(L * head_dim));
            V = (double *)malloc(sizeof(double) * (size_t)(L * head_dim));
            x = (double *)malloc(sizeof(double) * (size_t)(L + 1));
            qv = (double *)malloc(sizeof(double) * (size_t)head_dim);
        }
        for (int32_t g = 0; ok && C > 0 && g < num_kv_heads; ++g) {
            if (gather_sequence(k_pool, v_pool, row, L, g, num_kv_heads, head_dim, block_size,
                                num_blocks, is_bf16, K, V) != 0) {
                ok = 0;
                break;
            }
            for (int32_t hh = 0; hh < group; ++hh) {
                int32_t h = g * group + hh;
                for (int64_t j = 0; j < C; ++j) {
                    int64_t pos = L - C + j;
                    int64_t r = r0 + j;
                    for (int32_t d = 0; d < head_dim; ++d)
                        qv[d] = to_double(q[(r * num_q_heads + h) * head_dim + d], is_bf16);
                    attend_rows(qv, K, V, pos + 1, head_dim, scale, x,
                                out + (r * num_q_heads + h) * head_dim, NULL, NULL, NULL);
                }
            }
        }
        if (!ok) {
            ++bad;
            for (int64_t r = r0; r < r1 && C > 0; ++r)
                for (int64_t e = 0; e < (int64_t)num_q_heads * head_dim; ++e)
                    out[r * num_q_heads * head_dim + e] = 0.0;
        }
        free(K); free(V); free(x); free(qv);
    }
    return bad;
}

/* Gather a sequence's dequantized K/V (code * scale, exact in fp64) from an
 * 8-bit pool for kv head g.  Returns -1 when a table entry is outside the pool. */
static int gather_sequence_q8(const int8_t *k_codes, const int8_t *v_codes,
                              const uint16_t *k_scales, const uint16_t *v_scales,
                              const int32_t *table_row, int64_t n, int32_t g,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              int64_t num_blocks, double *K, double *V)
{
    int32_t ng = head_dim / 32;
    for (int64_t j = 0; j < n; ++j) {
        int64_t logical = j / block_size;          /* logical block of token j */
        int64_t block = table_row[logical];
        int64_t offset = j - logical * block_size;
        if (block >= num_blocks || block < 0) return -1;
        int64_t slab = block * num_kv_heads + g;
        for (int32_t d = 0; d < head_dim; ++d) {
            double ks = oracle_f16_to_double(k_scales[(slab * block_size + offset) * ng + d / 32]);
            double vs = oracle_f16_to_double(v_scales[(slab * block_size + offset) * ng + d / 32]);
            K[j * head_dim + d] = ks * k_codes[(slab * block_size + offset) * head_dim + d];
            V[j * head_dim + d] = vs * v_codes[(slab * head_dim + d) * block_size + offset];
        }
    }
    return 0;
}

/* PagedAttention decode over an 8-bit cache: the definition of
 * oracle_paged_decode with K and V taken as code * scale. */
int64_t oracle_paged_decode_q8(const uint16_t *q, const int8_t *k_codes, const int8_t *v_codes,
                               const uint16_t *k_scales, const uint16_t *v_scales,
                               const int32_t *block_tables, int32_t max_blocks_per_seq,
                               const int32_t *context_lens, int32_t num_seqs,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t block_size, int64_t num_blocks, int is_bf16,
                               double scale, double *out, int num_threads)
{
    int32_t group = num_q_heads / num_kv_heads;
    int64_t bad = 0;
    int64_t rows = (int64_t)num_seqs * num_q_heads;
#ifdef _OPENMP
    if (num_threads < 1) num_threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(+ : bad)
#endif
    for (int64_t r = 0; r < rows; ++r) {
        int32_t s = (int32_t)(r / num_q_heads), h = (int32_t)(r % num_q_heads);
        int32_t kv_head = h / group;
        int64_t n = context_lens[s];
        double *o = out + r * head_dim;
        if (n < 0 || n > (int64_t)block_size * max_blocks_per_seq) {
            for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
            if (h == 0) ++bad;
            continue;
        }
        double *K = (double *)malloc(sizeof(double) * (size_t)(n * head_dim + 1));
        double *V = (double *)malloc(sizeof(double) * (size_t)(n * head_dim + 1));
        double *x = (double *)malloc(sizeof(double) * (size_t)(n + 1));
        double *qv = (double *)malloc(sizeof(double) * (size_t)head_dim);
        const int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
        if (gather_sequence_q8(k_codes, v_codes, k_scales, v_scales, row, n, kv_head, num_kv_heads,
                               head_dim, block_size, num_blocks, K, V) != 0) {
            for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
            if (h == 0) ++bad;
        } else {
            for (int32_t d = 0; d < head_dim; ++d)
                qv[d] = to_double(q[r * head_dim + d], is_bf16);
            attend_rows(qv, K, V, n, head_dim, scale, x, o, NULL, NULL, NULL);
        }
        free(K); free(V); free(x); free(qv);
    }
    return bad;
}

/* One split of a sequence: attention pieces over logical tokens [t0, t1) of
 * sequence s, query head h: acc[D] = sum_j w_j v_j with w_j = exp(x_j - m),
 * m = max x_j, l = sum_j w_j.  An empty range gives m = -inf, l = 0, acc = 0. */
int oracle_paged_partial(const uint16_t *q, const uint16_t *k_pool,
                         const uint16_t *v_pool, const int32_t *block_tables,
                         int32_t max_blocks_per_seq, int32_t s, int32_t h,
                         int64_t t0, int64_t t1, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int64_t num_blocks, int is_bf16,
                         double scale, double *acc, double *m, double *l)
{
    int32_t g = h / (num_q_heads / num_kv_heads);
    int64_t n = t1 > t0 ? t1 - t0 : 0;
    const int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
    double *K = (double *)malloc(sizeof(double) * (size_t)((t1 > 0 ? t1 : 1) * head_dim));
    double *V = (double *)malloc(sizeof(double) * (size_t)((t1 > 0 ? t1 : 1) * head_dim));
    double *x = (double *)malloc(sizeof(double) * (size_t)(n + 1));
    double *qv = (double *)malloc(sizeof(double) * (size_t)head_dim);
    double *o = (double *)malloc(sizeof(double) * (size_t)head_dim);
    int rc = gather_sequence(k_pool, v_pool, row, t1, g, num_kv_heads, head_dim,
                             block_size, num_blocks, is_bf16, K, V);
    if (rc == 0) {
        for (int32_t d = 0; d < head_dim; ++d)
            qv[d] = to_double(q[((int64_t)s * num_q_heads + h) * head_dim + d], is_bf16);
        attend_rows(qv, K + t0 * head_dim, V + t0 * head_dim, n, head_dim, scale,
                    x, o, acc, m, l);
    }
    free(K); free(V); free(x); free(qv); free(o);
    return rc;
}

/* Log-sum-exp merge of P splits of one softmax:
 *   M = max_p m_p,  L = sum_p l_p e^{m_p - M},  out = sum_p acc_p e^{m_p - M} / L.
 * parts_acc [P][D], parts_m [P], parts_l [P]. */
void oracle_lse_merge(const double *parts_acc, const double *parts_m,
                      const double *parts_l, int32_t num_parts, int32_t head_dim,
                      double *out)
{
    double M = -INFINITY;
    for (int32_t p = 0; p < num_parts; ++p)
        if (parts_m[p] > M) M = parts_m[p];
    if (M == -INFINITY) {
        for (int32_t d = 0; d < head_dim; ++d) out[d] = 0.0;
        return;
    }
    double L = 0.0;
    for (int32_t p = 0; p < num_parts; ++p)
        if (parts_l[p] > 0.0) L += parts_l[p] * exp(parts_m[p] - M);
    for (int32_t d = 0; d < head_dim; ++d) {
        double a = 0.0;
        for (int32_t p = 0; p < num_parts; ++p)
            if (parts_l[p] > 0.0) a += parts_acc[(int64_t)p * head_dim + d] * exp(parts_m[p] - M);
        out[d] = a / L;
    }
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
