/*
 * ns_oracle.c -- fp64 CPU oracle for the paged-KV hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file.  Only the tests, the package smoke check and the benchmark's
 * CPU-baseline / reference arm use it.  It shares no code, header, table or
 * constant with the CUDA library: its element decoders, indexing and
 * arithmetic are written out here from the definitions below.
 *
 * What it computes (the plain definitions, no blocking, no online softmax):
 *
 *  kv_append -- each step stores its tokens' new K/V rows in the cache
 *    (Inference Engineering Day 11 short, "How does vLLM work"); with the paged layout of the nanoserve project page ("What I
 *    built", paged KV cache bullet) a token's slot s lives in block s / bs at
 *    offset s % bs.  Pool layout [num_blocks][Hkv][bs][D].  A negative slot
 *    marks a padding token and is skipped.  Pure copy of bit patterns.
 *
 *  paged_attention -- every query head of every sequence attends over that
 *    sequence's cached keys, found through its block table (nanoserve
 *    project page, "What I built", fused paged-attention decode bullet: online
 *    softmax over the block table; online softmax is an exact reformulation
 *    of softmax, so the oracle evaluates softmax directly):
 *        kv head of q head j      h = j / (Hq / Hkv)
 *        key position p           block = table[s][p / bs], offset p % bs
 *        score                    z_p = scale * sum_d q[j][d] * K[p][d]
 *        weights                  w_p = exp(z_p - max z) / sum_p' exp(z_p' - max z)
 *        output                   o[d] = sum_p w_p * V[p][d]
 *    Query token i of a span of q_len tokens in a sequence of L tokens sits
 *    at position L - q_len + i and sees keys p <= L - q_len + i (cached
 *    prefix plus causal within the chunk: Inference Engineering Day 12 short,
 *    "What is chunked prefill within vLLM").  A decode step is the span
 *    q_len = 1, which sees all L keys.  A query that sees no key (L = 0)
 *    yields o = 0.
 *
 * Everything is evaluated in double precision from the exact values of the
 * fp16 / bf16 inputs; the result is returned unrounded as double.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F16 0
#define ORACLE_BF16 1

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);              /* subnormal: f * 2^(1-15-10) */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);  /* (1 + f/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);             /* subnormal: f * 2^(1-127-7) */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);  /* (1 + f/2^7) * 2^(e-127) */
    return sign ? -v : v;
}

static double elem(int dtype, uint16_t bits)
{
    return dtype == ORACLE_BF16 ? oracle_bf16_to_double(bits) : oracle_f16_to_double(bits);
}

/*
 * Copy each token's K and V rows into its pool slot.
 *   k, v          [num_tokens][Hkv][D]
 *   slot_mapping  [num_tokens]
 *   k_pool/v_pool [num_blocks][Hkv][bs][D]  (updated in place)
 * Returns 0, or -1 if a slot lies beyond the pool.
 */
int oracle_kv_append(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping,
                     uint16_t *k_pool, uint16_t *v_pool, int64_t num_tokens,
                     int num_kv_heads, int head_dim, int block_size, int64_t num_blocks)
{
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_blocks * (int64_t)block_size)
            return -1;
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int d = 0; d < head_dim; ++d) {
                int64_t src = (t * num_kv_heads + h) * head_dim + d;
                int64_t dst = ((block * num_kv_heads + h) * block_size + offset) * head_dim + d;
                k_pool[dst] = k[src];
                v_pool[dst] = v[src];
            }
        }
    }
    return 0;
}

/*
 * Attention of every query row over its sequence's paged keys.
 *   q               [num_q_rows][Hq][D]
 *   query_start_loc [num_seqs + 1] or NULL; NULL means one query row per
 *                   sequence (row s belongs to sequence s, a decode step)
 *   block_tables    [num_seqs][max_blocks_per_seq]
 *   context_lens    [num_seqs]  keys of each sequence, query tokens included
 *   out             [num_q_rows][Hq][D] double (written)
 * num_threads > 1 spreads the independent (row, head) problems over OpenMP
 * threads when the library was built with OpenMP; the arithmetic of each
 * problem is the same either way.
 * Returns 0, -1 for a block id outside the pool, -2 for bad lengths,
 * -3 for out of memory.
 */
int oracle_paged_attention(int dtype, const uint16_t *q, const int32_t *query_start_loc,
                           const uint16_t *k_pool, const uint16_t *v_pool,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *context_lens, int num_seqs,
                           int num_q_heads, int num_kv_heads, int head_dim,
                           int block_size, int64_t num_blocks, double scale,
                           double *out, int num_threads)
{
    if (num_q_heads % num_kv_heads != 0)
        return -2;
    int group = num_q_heads / num_kv_heads;

    /* Flatten the work into (query row, head) problems. */
    int64_t num_rows = query_start_loc ? query_start_loc[num_seqs] : num_seqs;
    int64_t *row_seq = (int64_t *)malloc(sizeof(int64_t) * (size_t)(num_rows > 0 ? num_rows : 1));
    int64_t *row_pos = (int64_t *)malloc(sizeof(int64_t) * (size_t)(num_rows > 0 ? num_rows : 1));
    if (!row_seq || !row_pos) {
        free(row_seq);
        free(row_pos);
        return -3;
    }
    for (int s = 0; s < num_seqs; ++s) {
        int64_t first = query_start_loc ? query_start_loc[s] : s;
        int64_t q_len = query_start_loc ? query_start_loc[s + 1] - query_start_loc[s] : 1;
        int64_t L = context_lens[s];
        if (q_len < 0 || L < 0 || q_len > (L > 0 ? L : 1) ||
            L > (int64_t)max_blocks_per_seq * block_size) {
            free(row_seq);
            free(row_pos);
            return -2;
        }
        for (int64_t i = 0; i < q_len; ++i) {
            row_seq[first + i] = s;
            row_pos[first + i] = L - q_len + i;   /* absolute position of the query token */
        }
    }

    int err = 0;
    int64_t num_problems = num_rows * num_q_heads;
#ifdef _OPENMP
    if (num_threads < 1)
        num_threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
    for (int64_t prob = 0; prob < num_problems; ++prob) {
        int64_t row = prob / num_q_heads;
        int j = (int)(prob % num_q_heads);
        int64_t s = row_seq[row];
        int64_t n_keys = row_pos[row] + 1;       /* keys 0 .. position */
        if (context_lens[s] == 0)
            n_keys = 0;
        int h = j / group;
        double *o = out + (row * num_q_heads + j) * head_dim;
        for (int d = 0; d < head_dim; ++d)
            o[d] = 0.0;
        if (n_keys <= 0)
            continue;

        double *z = (double *)malloc(sizeof(double) * (size_t)n_keys);
        double *qv = (double *)malloc(sizeof(double) * (size_t)head_dim);
        if (!z || !qv) {
            free(z);
            free(qv);
#ifdef _OPENMP
#pragma omp atomic write
#endif
            err = -3;
            continue;
        }
        for (int d = 0; d < head_dim; ++d)
            qv[d] = elem(dtype, q[(row * num_q_heads + j) * head_dim + d]);

        /* Scores through the block table. */
        int bad = 0;
        for (int64_t p = 0; p < n_keys; ++p) {
            int64_t block = block_tables[s * (int64_t)max_blocks_per_seq + p / block_size];
            if (block < 0 || block >= num_blocks) {
                bad = 1;
                break;
            }
            const uint16_t *kr = k_pool + ((block * num_kv_heads + h) * block_size + p % block_size) * head_dim;
            double dot = 0.0;
            for (int d = 0; d < head_dim; ++d)
                dot += qv[d] * elem(dtype, kr[d]);
            z[p] = scale * dot;
        }
        if (bad) {
            free(z);
            free(qv);
#ifdef _OPENMP
#pragma omp atomic write
#endif
            err = -1;
            continue;
        }

        /* Softmax. */
        double zmax = z[0];
        for (int64_t p = 1; p < n_keys; ++p)
            if (z[p] > zmax)
                zmax = z[p];
        double denom = 0.0;
        for (int64_t p = 0; p < n_keys; ++p) {
            z[p] = exp(z[p] - zmax);
            denom += z[p];
        }

        /* Weighted sum of values. */
        for (int64_t p = 0; p < n_keys; ++p) {
            int64_t block = block_tables[s * (int64_t)max_blocks_per_seq + p / block_size];
            const uint16_t *vr = v_pool + ((block * num_kv_heads + h) * block_size + p % block_size) * head_dim;
            double w = z[p] / denom;
            for (int d = 0; d < head_dim; ++d)
                o[d] += w * elem(dtype, vr[d]);
        }
        free(z);
        free(qv);
    }
    free(row_seq);
    free(row_pos);
    return err;
}

/* Number of OpenMP threads the library would use (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
