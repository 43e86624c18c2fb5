/*
 * ORACLE -- test infrastructure only.  Nothing in the product path may link,
 * load or call this file; only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark do.
 *
 * Plain CPU definition of single-query paged decode attention, in fp64.
 *
 * What it computes (PagedAttention notes, unpurerationalist.github.io, §3.1,
 * the blockwise attention equation; the same equation in the vLLM paper
 * review, mz-moonzoo.tistory.com/116, §4.1, whose denominator is garbled
 * there and is read as the double sum over all valid tokens of all blocks):
 *
 *   for the query q_i of a sequence, with its keys and values split into
 *   blocks K_j, V_j of B tokens,
 *     A_ij = exp(q_i K_j^T / sqrt(d)) / sum_t sum_s exp(q_i k_ts^T / sqrt(d))
 *     o_i  = sum_j A_ij V_j
 *
 * which is ordinary softmax attention over the sequence's valid tokens.
 * Token position p lives in logical block p / B at offset p % B, and the
 * block table maps that logical block to a physical block (paged KV cache
 * tutorial, llm-systems-engineering.pages.dev/posts/paged-kv-cache, Fig. 2,
 * "position 6 -> L1 offset 2 -> P0").  Only the first ctx_len positions are
 * valid; unwritten slots of the last block take no part (same tutorial,
 * Fig. 4).  The context includes the token written in this decode step
 * (Fig. 4: the query at position 8 uses positions 0..8).
 *
 * Cache byte layout read here (a data format, not code shared with anything):
 *   cache[num_blocks][num_heads][block_size][head_dim], IEEE binary16 values.
 *
 * The scale is passed in (1/sqrt(d) in the pages).  The softmax is evaluated
 * as exp(x_j - max x) / sum exp(x - max x), which is the same real number as
 * the pages' ratio; fp64 throughout.  A context length of 0 gives o = 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16 -> double, from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; exponent 0 is
 * subnormal (fraction * 2^-24), exponent 31 is inf / nan. */
static double half_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24);
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(frac | 0x400), expo - 25);
    }
    return sign ? -mag : mag;
}

static double g_half_table[65536];
static int g_half_table_ready = 0;

static void build_half_table(void)
{
    if (g_half_table_ready) return;
    for (int i = 0; i < 65536; ++i) g_half_table[i] = half_bits_to_double((uint16_t)i);
    g_half_table_ready = 1;
}

double oracle_half_to_double(uint16_t h) { return half_bits_to_double(h); }

/* Returns 0 on success, -1 on a bad argument, -2 if a block table entry that
 * covers a valid position is outside [0, num_blocks). */
int oracle_paged_attention(double *out,                  /* [S][H][D]            */
                           const uint16_t *q,            /* [S][H][D]  fp16 bits */
                           const uint16_t *k_cache,      /* [NB][H][B][D]        */
                           const uint16_t *v_cache,      /* [NB][H][B][D]        */
                           const int32_t *block_tables,  /* [S][max_blocks]      */
                           const int32_t *ctx_lens,      /* [S]                  */
                           int32_t S, int32_t H, int32_t D, int32_t B,
                           int32_t num_blocks, int32_t max_blocks,
                           double scale, int32_t num_threads)
{
    if (S < 0 || H <= 0 || D <= 0 || B <= 0 || num_blocks < 0 || max_blocks < 0) return -1;
    for (int32_t s = 0; s < S; ++s) {
        int32_t n = ctx_lens[s];
        if (n < 0 || (int64_t)n > (int64_t)max_blocks * B) return -1;
        for (int32_t j = 0; j < (n + B - 1) / B; ++j) {
            int32_t blk = block_tables[(int64_t)s * max_blocks + j];
            if (blk < 0 || blk >= num_blocks) return -2;
        }
    }
    build_half_table();
    int64_t pairs = (int64_t)S * H;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif
#pragma omp parallel
    {
        double *x = NULL;   /* scores of the valid tokens      */
        int32_t x_cap = 0;
#pragma omp for schedule(dynamic, 4)
        for (int64_t pair = 0; pair < pairs; ++pair) {
            int32_t s = (int32_t)(pair / H);
            int32_t h = (int32_t)(pair % H);
            int32_t n = ctx_lens[s];
            double *o = out + pair * D;
            for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
            if (n == 0) continue;
            if (n > x_cap) {
                free(x);
                x_cap = n;
                x = (double *)malloc(sizeof(double) * (size_t)n);
            }
            const uint16_t *qv = q + pair * D;
            /* scores x_p = (q . k_p) * scale for every valid position p */
            double m = -INFINITY;
            for (int32_t p = 0; p < n; ++p) {
                int32_t blk = block_tables[(int64_t)s * max_blocks + p / B];
                int32_t off = p % B;
                const uint16_t *kv = k_cache + (((int64_t)blk * H + h) * B + off) * D;
                double dot = 0.0;
                for (int32_t d = 0; d < D; ++d) dot += g_half_table[qv[d]] * g_half_table[kv[d]];
                x[p] = dot * scale;
                if (x[p] > m) m = x[p];
            }
            /* A_p = exp(x_p - m) / sum exp(x - m);  o = sum_p A_p v_p */
            double denom = 0.0;
            for (int32_t p = 0; p < n; ++p) {
                x[p] = exp(x[p] - m);
                denom += x[p];
            }
            for (int32_t p = 0; p < n; ++p) {
                int32_t blk = block_tables[(int64_t)s * max_blocks + p / B];
                int32_t off = p % B;
                const uint16_t *vv = v_cache + (((int64_t)blk * H + h) * B + off) * D;
                double a = x[p] / denom;
                for (int32_t d = 0; d < D; ++d) o[d] += a * g_half_table[vv[d]];
            }
        }
        free(x);
    }
    return 0;
}

/* Paged prefill (many queries per sequence, causal): the queries of
 * sequence s are rows q_starts[s] .. q_starts[s+1]-1 of q and are the last
 * q_len = q_starts[s+1] - q_starts[s] positions of its context of ctx_lens[s]
 * tokens; the query at position p attends to positions 0..p (the paper
 * review's §4.3 prompt phase: every prompt token attends to the tokens
 * before it and itself).  Same blockwise softmax as the decode oracle.
 * out: [T][H][D] fp64, T = q_starts[S].  Returns 0, -1 on a bad argument,
 * -2 on a table entry outside the pool. */
int oracle_paged_prefill(double *out, const uint16_t *q, const uint16_t *k_cache,
                         const uint16_t *v_cache, const int32_t *block_tables,
                         const int32_t *ctx_lens, const int32_t *q_starts, int32_t S, int32_t H,
                         int32_t D, int32_t B, int32_t num_blocks, int32_t max_blocks,
                         double scale, int32_t num_threads)
{
    if (S < 0 || H <= 0 || D <= 0 || B <= 0 || max_blocks < 0) return -1;
    if (S > 0 && q_starts[0] != 0) return -1;
    for (int32_t s = 0; s < S; ++s) {
        int32_t n = ctx_lens[s], ql = q_starts[s + 1] - q_starts[s];
        if (n < 0 || ql < 0 || ql > n || (int64_t)n > (int64_t)max_blocks * B) return -1;
        for (int32_t j = 0; j < (n + B - 1) / B; ++j) {
            int32_t blk = block_tables[(int64_t)s * max_blocks + j];
            if (blk < 0 || blk >= num_blocks) return -2;
        }
    }
    build_half_table();
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif
    int64_t T = S > 0 ? q_starts[S] : 0;
#pragma omp parallel
    {
        double *x = NULL;
        int32_t x_cap = 0;
#pragma omp for schedule(dynamic, 8)
        for (int64_t item = 0; item < T * H; ++item) {
            int64_t row = item / H;
            int32_t h = (int32_t)(item % H);
            int32_t s = 0;                          /* sequence owning this row */
            while (q_starts[s + 1] <= row) ++s;
            int32_t n = ctx_lens[s];
            int32_t ql = q_starts[s + 1] - q_starts[s];
            int32_t pos = n - ql + (int32_t)(row - q_starts[s]);
            int32_t m_tok = pos + 1;                /* causal: positions 0..pos */
            double *o = out + item * D;
            for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
            if (m_tok > x_cap) {
                free(x);
                x_cap = m_tok;
                x = (double *)malloc(sizeof(double) * (size_t)m_tok);
            }
            const uint16_t *qv = q + item * D;
            double mx = -INFINITY;
            for (int32_t p = 0; p < m_tok; ++p) {
                int32_t blk = block_tables[(int64_t)s * max_blocks + p / B];
                const uint16_t *kv = k_cache + (((int64_t)blk * H + h) * B + p % B) * D;
                double dot = 0.0;
                for (int32_t d = 0; d < D; ++d) dot += g_half_table[qv[d]] * g_half_table[kv[d]];
                x[p] = dot * scale;
                if (x[p] > mx) mx = x[p];
            }
            double denom = 0.0;
            for (int32_t p = 0; p < m_tok; ++p) {
                x[p] = exp(x[p] - mx);
                denom += x[p];
            }
            for (int32_t p = 0; p < m_tok; ++p) {
                int32_t blk = block_tables[(int64_t)s * max_blocks + p / B];
                const uint16_t *vv = v_cache + (((int64_t)blk * H + h) * B + p % B) * D;
                double a = x[p] / denom;
                for (int32_t d = 0; d < D; ++d) o[d] += a * g_half_table[vv[d]];
            }
        }
        free(x);
    }
    return 0;
}

/* Threads an OpenMP parallel region would use (for reporting the CPU
 * baseline's core count). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
