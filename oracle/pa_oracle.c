/*
 * pa_oracle.c -- CPU oracle for paged-attention decode and reshape_and_cache.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and
 * the benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header or constant with the CUDA library: it is a plain, slow restatement of
 * what the pages define, computed in fp64, so a reader can check it by eye.
 *
 * What it computes (sources: the pages on vLLM):
 *
 *  - Decode attention: o_t = Attention(q_t, K_{1:t}, V_{1:t}), one query per
 *    head over that sequence's whole K/V history
 *    ("vLLM 2026 推理引擎全解", §1.1), i.e. o = softmax(scale * K q)^T V.
 *  - The history lives in fixed blocks of block_size tokens, reached through a
 *    per-sequence block table (logical block -> physical block); paging only
 *    changes addressing, attention itself does not see it
 *    ("vLLM 2026 推理引擎全解", §2.1; mjmagnets.cn vLLM tutorial, §2.2: the
 *    operator gathers the K and V blocks through the table, then computes).
 *  - Cache layout [num_blocks, num_heads, block_size, head_dim]
 *    ("vLLM 2026 推理引擎全解", §2.2, kernel sketch).
 *  - reshape_and_cache stores each new token's K and V into its slot, where
 *    slot = physical_block * block_size + offset; a negative slot is skipped
 *    (the pages name the step -- "append new token", doramagic.ai vLLM manual,
 *    "KVCacheManager 缓存管理" -- but not the encoding; this is the plainest
 *    reading).
 *
 * So the oracle, per (sequence s, head h):
 *   1. gathers K_s, V_s (ctx_s x head_dim) through the block table, converting
 *      each fp16 (or bf16) value exactly to double;
 *   2. scores_t = scale * sum_d q[d] * K_s[t][d];
 *   3. weights_t = exp(scores_t - max_t scores_t), normalised by their sum;
 *   4. out[d] = sum_t weights_t * V_s[t][d].
 * A sequence with ctx_s == 0 gets a zero output.
 *
 * Parity of every function here is pinned by the CPU tests against facts the
 * pages and the mathematics fix (brute force, closed forms, invariances, and
 * an fp64 library attention), not against this file.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG -1
#define ORACLE_BAD_CONTEXT -2
#define ORACLE_BAD_TABLE -3
#define ORACLE_BAD_SLOT -4
#define ORACLE_NO_MEMORY -5

/* IEEE 754 binary16 -> double, exactly, from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int exponent = (bits >> 10) & 0x1f;
    int fraction = bits & 0x3ff;
    double magnitude;
    if (exponent == 0) {
        magnitude = ldexp((double)fraction, -24);            /* subnormal or zero */
    } else if (exponent == 31) {
        magnitude = fraction ? NAN : INFINITY;
    } else {
        magnitude = ldexp((double)(1024 + fraction), exponent - 25);
    }
    return sign ? -magnitude : magnitude;
}

/* bfloat16 -> double, exactly: a bfloat16 is the upper 16 bits of an IEEE
 * 754 binary32 (1 sign bit, 8 exponent bits, 7 fraction bits). */
double oracle_bf16_to_double(uint16_t bits)
{
    uint32_t word = (uint32_t)bits << 16;
    float value;
    memcpy(&value, &word, sizeof value);
    return (double)value;
}

#define ORACLE_F16 0
#define ORACLE_BF16 1

static double element_to_double(uint16_t bits, int dtype)
{
    return dtype == ORACLE_BF16 ? oracle_bf16_to_double(bits) : oracle_half_to_double(bits);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Offset of element (block, head, token-in-block, dim) in a
 * [num_blocks, num_heads, block_size, head_dim] cache. */
static size_t cache_index(int64_t block, int head, int offset, int dim,
                          int num_heads, int block_size, int head_dim)
{
    return (((size_t)block * (size_t)num_heads + (size_t)head) * (size_t)block_size
            + (size_t)offset) * (size_t)head_dim + (size_t)dim;
}

/*
 * Decode attention for every (sequence, head).
 *
 * out           [num_seqs, num_heads, head_dim] double (written)
 * q             [num_seqs, num_heads, head_dim] 16-bit element bits
 * k_cache       [num_blocks, num_heads, block_size, head_dim] element bits
 * v_cache       same layout as k_cache
 * dtype         0: elements are IEEE binary16; 1: bfloat16
 * block_tables  [num_seqs, max_blocks_per_seq] int32
 * context_lens  [num_seqs] int32
 *
 * Returns ORACLE_OK, or a negative code if a context length or a used table
 * entry is out of range (nothing is computed then).
 */
int oracle_decode(double *out, const uint16_t *q, const uint16_t *k_cache,
                  const uint16_t *v_cache, const int32_t *block_tables,
                  const int32_t *context_lens, double scale, int num_seqs,
                  int num_heads, int head_dim, int block_size, int num_blocks,
                  int max_blocks_per_seq, int dtype)
{
    if (num_seqs < 0 || num_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks < 0 || max_blocks_per_seq <= 0 ||
        (dtype != ORACLE_F16 && dtype != ORACLE_BF16))
        return ORACLE_BAD_ARG;

    /* Check every input the computation will use before computing anything. */
    for (int s = 0; s < num_seqs; ++s) {
        int ctx = context_lens[s];
        if (ctx < 0 || (int64_t)ctx > (int64_t)max_blocks_per_seq * block_size)
            return ORACLE_BAD_CONTEXT;
        int used_blocks = (ctx + block_size - 1) / block_size;
        for (int b = 0; b < used_blocks; ++b) {
            int32_t phys = block_tables[(size_t)s * max_blocks_per_seq + b];
            if (phys < 0 || phys >= num_blocks)
                return ORACLE_BAD_TABLE;
        }
    }

    int failed = 0;
    int num_pairs = num_seqs * num_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int pair = 0; pair < num_pairs; ++pair) {
        int s = pair / num_heads;
        int h = pair % num_heads;
        int ctx = context_lens[s];
        double *o = out + (size_t)pair * head_dim;
        for (int d = 0; d < head_dim; ++d)
            o[d] = 0.0;
        if (ctx == 0)
            continue;

        double *K = malloc(sizeof(double) * (size_t)ctx * head_dim);
        double *V = malloc(sizeof(double) * (size_t)ctx * head_dim);
        double *qd = malloc(sizeof(double) * (size_t)head_dim);
        double *weights = malloc(sizeof(double) * (size_t)ctx);
        if (!K || !V || !qd || !weights) {
            free(K); free(V); free(qd); free(weights);
#pragma omp atomic write
            failed = 1;
            continue;
        }

        /* Step 1: gather this sequence's K and V through its block table into
         * contiguous [ctx, head_dim] arrays (logical token t lives in logical
         * block t / block_size at offset t % block_size). */
        for (int t = 0; t < ctx; ++t) {
            int64_t phys = block_tables[(size_t)s * max_blocks_per_seq + t / block_size];
            int offset = t % block_size;
            for (int d = 0; d < head_dim; ++d) {
                size_t at = cache_index(phys, h, offset, d, num_heads, block_size, head_dim);
                K[(size_t)t * head_dim + d] = element_to_double(k_cache[at], dtype);
                V[(size_t)t * head_dim + d] = element_to_double(v_cache[at], dtype);
            }
        }
        for (int d = 0; d < head_dim; ++d)
            qd[d] = element_to_double(q[(size_t)pair * head_dim + d], dtype);

        /* Step 2: scaled scores. */
        double max_score = -INFINITY;
        for (int t = 0; t < ctx; ++t) {
            double dot = 0.0;
            for (int d = 0; d < head_dim; ++d)
                dot += qd[d] * K[(size_t)t * head_dim + d];
            weights[t] = scale * dot;
            if (weights[t] > max_score)
                max_score = weights[t];
        }

        /* Step 3: softmax, with the maximum subtracted before exp. */
        double total = 0.0;
        for (int t = 0; t < ctx; ++t) {
            weights[t] = exp(weights[t] - max_score);
            total += weights[t];
        }

        /* Step 4: weighted sum of the value rows. */
        for (int t = 0; t < ctx; ++t) {
            double w = weights[t] / total;
            for (int d = 0; d < head_dim; ++d)
                o[d] += w * V[(size_t)t * head_dim + d];
        }

        free(K); free(V); free(qd); free(weights);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * reshape_and_cache: for each new token i with slot_mapping[i] >= 0, copy
 * k[i, h, :] and v[i, h, :] into k_cache / v_cache at
 * (slot / block_size, h, slot % block_size, :) for every head h.
 *
 * k, v          [num_tokens, num_heads, head_dim] fp16 bits
 * k_cache, ...  [num_blocks, num_heads, block_size, head_dim] fp16 bits (updated)
 *
 * Returns ORACLE_BAD_SLOT, without writing anything, if a slot is past the
 * end of the pool.
 */
int oracle_reshape_and_cache(const uint16_t *k, const uint16_t *v, uint16_t *k_cache,
                             uint16_t *v_cache, const int32_t *slot_mapping,
                             int num_tokens, int num_heads, int head_dim,
                             int block_size, int num_blocks)
{
    if (num_tokens < 0 || num_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks < 0)
        return ORACLE_BAD_ARG;
    for (int i = 0; i < num_tokens; ++i)
        if ((int64_t)slot_mapping[i] >= (int64_t)num_blocks * block_size)
            return ORACLE_BAD_SLOT;

    for (int i = 0; i < num_tokens; ++i) {
        int32_t slot = slot_mapping[i];
        if (slot < 0)
            continue;
        int64_t block = slot / block_size;
        int offset = slot % block_size;
        for (int h = 0; h < num_heads; ++h) {
            for (int d = 0; d < head_dim; ++d) {
                size_t src = ((size_t)i * num_heads + h) * head_dim + d;
                size_t dst = cache_index(block, h, offset, d, num_heads, block_size, head_dim);
                k_cache[dst] = k[src];
                v_cache[dst] = v[src];
            }
        }
    }
    return ORACLE_OK;
}

/*
 * copy_blocks: for each pair (src, dst) of block_pairs [num_pairs][2], copy K
 * and V of block src of the source pool, every head, to block dst of the
 * destination pool -- the KV cache manager's block copy and CPU swap
 * (doramagic.ai vLLM manual, "内存管理策略", "BlockPool 组件").
 *
 * Pools are [num_blocks, num_heads, block_size, head_dim] 16-bit elements.
 * Returns ORACLE_BAD_TABLE, without copying anything, if an id is out of its
 * pool.
 */
int oracle_copy_blocks(const uint16_t *src_k, const uint16_t *src_v, int src_num_blocks,
                       uint16_t *dst_k, uint16_t *dst_v, int dst_num_blocks,
                       const int32_t *block_pairs, int num_pairs, int num_heads, int head_dim,
                       int block_size)
{
    if (num_pairs < 0 || num_heads <= 0 || head_dim <= 0 || block_size <= 0)
        return ORACLE_BAD_ARG;
    for (int i = 0; i < num_pairs; ++i) {
        int32_t src = block_pairs[2 * i], dst = block_pairs[2 * i + 1];
        if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks)
            return ORACLE_BAD_TABLE;
    }
    for (int i = 0; i < num_pairs; ++i) {
        int64_t src = block_pairs[2 * i], dst = block_pairs[2 * i + 1];
        for (int h = 0; h < num_heads; ++h)
            for (int t = 0; t < block_size; ++t)
                for (int d = 0; d < head_dim; ++d) {
                    size_t from = cache_index(src, h, t, d, num_heads, block_size, head_dim);
                    size_t to = cache_index(dst, h, t, d, num_heads, block_size, head_dim);
                    dst_k[to] = src_k[from];
                    dst_v[to] = src_v[from];
                }
    }
    return ORACLE_OK;
}

/*
 * Paged prefill: causal multi-query attention over the paged cache.
 *
 * Sequence s has q_len_s = query_start[s + 1] - query_start[s] query rows
 * (rows query_start[s] .. query_start[s + 1] - 1 of q and out), which are the
 * last q_len_s tokens of its context: query i sits at position
 * p = ctx_s - q_len_s + i and attends to keys 0 .. p of the sequence
 * ("vLLM 2026 推理引擎全解", §1.3: prefill processes the prompt, computing many
 * positions at once; §1.1: o_t = Attention(q_t, K_{1:t}, V_{1:t}) for each t).
 * Their K/V are already in the cache.
 *
 * out          [total_q, num_heads, head_dim] double (written)
 * q            [total_q, num_heads, head_dim] 16-bit element bits
 * query_start  [num_seqs + 1] int32, non-decreasing, query_start[0] = 0
 * Other arrays and dtype as oracle_decode.  Returns ORACLE_BAD_CONTEXT if a
 * sequence has more queries than tokens.
 */
int oracle_prefill(double *out, const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                   const int32_t *block_tables, const int32_t *context_lens,
                   const int32_t *query_start, double scale, int num_seqs, int num_heads,
                   int head_dim, int block_size, int num_blocks, int max_blocks_per_seq, int dtype)
{
    if (num_seqs < 0 || num_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks < 0 || max_blocks_per_seq <= 0 ||
        (dtype != ORACLE_F16 && dtype != ORACLE_BF16) || (num_seqs > 0 && query_start[0] != 0))
        return ORACLE_BAD_ARG;
    for (int s = 0; s < num_seqs; ++s) {
        int ctx = context_lens[s];
        int q_len = query_start[s + 1] - query_start[s];
        if (ctx < 0 || (int64_t)ctx > (int64_t)max_blocks_per_seq * block_size || q_len < 0 ||
            q_len > ctx)
            return ORACLE_BAD_CONTEXT;
        for (int b = 0; b < (ctx + block_size - 1) / block_size; ++b) {
            int32_t phys = block_tables[(size_t)s * max_blocks_per_seq + b];
            if (phys < 0 || phys >= num_blocks)
                return ORACLE_BAD_TABLE;
        }
    }

    int failed = 0;
    int num_pairs = num_seqs * num_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int pair = 0; pair < num_pairs; ++pair) {
        int s = pair / num_heads;
        int h = pair % num_heads;
        int ctx = context_lens[s];
        int q_first = query_start[s];
        int q_len = query_start[s + 1] - q_first;
        if (q_len == 0)
            continue;
        double *K = malloc(sizeof(double) * (size_t)ctx * head_dim);
        double *V = malloc(sizeof(double) * (size_t)ctx * head_dim);
        double *qd = malloc(sizeof(double) * (size_t)head_dim);
        double *weights = malloc(sizeof(double) * (size_t)ctx);
        if (!K || !V || !qd || !weights) {
            free(K); free(V); free(qd); free(weights);
#pragma omp atomic write
            failed = 1;
            continue;
        }
        /* gather the sequence's K and V through its block table */
        for (int t = 0; t < ctx; ++t) {
            int64_t phys = block_tables[(size_t)s * max_blocks_per_seq + t / block_size];
            int offset = t % block_size;
            for (int d = 0; d < head_dim; ++d) {
                size_t at = cache_index(phys, h, offset, d, num_heads, block_size, head_dim);
                K[(size_t)t * head_dim + d] = element_to_double(k_cache[at], dtype);
                V[(size_t)t * head_dim + d] = element_to_double(v_cache[at], dtype);
            }
        }
        for (int i = 0; i < q_len; ++i) {
            size_t row = ((size_t)(q_first + i) * num_heads + h) * head_dim;
            int pos = ctx - q_len + i;               /* this query's position */
            for (int d = 0; d < head_dim; ++d)
                qd[d] = element_to_double(q[row + d], dtype);
            double max_score = -INFINITY;
            for (int t = 0; t <= pos; ++t) {          /* causal: keys 0 .. pos */
                double dot = 0.0;
                for (int d = 0; d < head_dim; ++d)
                    dot += qd[d] * K[(size_t)t * head_dim + d];
                weights[t] = scale * dot;
                if (weights[t] > max_score)
                    max_score = weights[t];
            }
            double total = 0.0;
            for (int t = 0; t <= pos; ++t) {
                weights[t] = exp(weights[t] - max_score);
                total += weights[t];
            }
            for (int d = 0; d < head_dim; ++d)
                out[row + d] = 0.0;
            for (int t = 0; t <= pos; ++t) {
                double w = weights[t] / total;
                for (int d = 0; d < head_dim; ++d)
                    out[row + d] += w * V[(size_t)t * head_dim + d];
            }
        }
        free(K); free(V); free(qd); free(weights);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}
