/*
 * Plain fp64 CPU oracle for paged decode attention, the KV-cache slot
 * write and the whole-block copy.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test-suite, the package smoke check and the
 * benchmark's CPU-baseline / reference arm use it.  It shares no code,
 * header, table or helper with the CUDA library.
 *
 * Everything here is written for a reader to check by eye against the
 * definitions on the source pages; there is no blocking, fusion or
 * reordering beyond what those definitions state.
 *
 * Storage convention (the plainest reading of "separate key and value
 * caches" with "2048 elements per head per block" at block size 16 and
 * head size 128, vLLM PagedAttention & continuous batching, "The kernel
 * page"):
 *     k_cache, v_cache : [num_blocks][num_kv_heads][block_size][head_dim]
 * so the row of token slot `o` of physical block `b`, KV head `h`, starts at
 *     ((b * num_kv_heads + h) * block_size + o) * head_dim.
 * Scalars are stored as IEEE binary16 (dtype 0) or bfloat16 (dtype 1) bit
 * patterns and are widened to binary64 exactly before any arithmetic.  The
 * 8-bit cache variant stores one-byte E4M3 codes with one scale factor per
 * pool (see the FP8 section below).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_BAD_INDEX (-2)
#define ORACLE_NO_MEMORY (-3)

/* ------------------------------------------------------------------ */
/* Exact widening of 16-bit storage formats to binary64.               */
/* ------------------------------------------------------------------ */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Subnormals are fraction * 2^-24; normals are
 * (1024 + fraction) * 2^(exponent - 25). */
double oracle_f16_to_f64(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int exponent = (bits >> 10) & 0x1f;
    int fraction = bits & 0x3ff;
    double magnitude;
    if (exponent == 0) {
        magnitude = ldexp((double)fraction, -24);
    } else if (exponent == 31) {
        magnitude = fraction ? NAN : INFINITY;
    } else {
        magnitude = ldexp((double)(1024 + fraction), exponent - 25);
    }
    return sign ? -magnitude : magnitude;
}

/* bfloat16 is the upper half of an IEEE binary32 pattern. */
double oracle_bf16_to_f64(uint16_t bits) {
    uint32_t word = ((uint32_t)bits) << 16;
    float value;
    memcpy(&value, &word, sizeof value);
    return (double)value;
}

static double widen(uint16_t bits, int dtype) {
    return dtype == 0 ? oracle_f16_to_f64(bits) : oracle_bf16_to_f64(bits);
}

/* ------------------------------------------------------------------ */
/* FP8 E4M3 (the OCP 8-bit floating-point E4M3 encoding): 1 sign bit, 4  */
/* exponent bits with bias 7, 3 mantissa bits, no infinities; exponent   */
/* 15 with mantissa 7 is NaN, so the largest finite magnitude is         */
/* 1.75 * 2^8 = 448.  Exponent 0 holds the subnormals mantissa * 2^-9.   */
/* The pages say only that changing the key-value precision changes the  */
/* numerics ("Serving Language Models Within a Memory Budget", section 4); */
/* the reading used here: a pool stores code = E4M3(x / scale), rounded   */
/* from the binary32 quotient, and reads back code * scale.               */
/* ------------------------------------------------------------------ */
double oracle_e4m3_to_f64(uint8_t code) {
    int sign = code >> 7;
    int exponent = (code >> 3) & 0xf;
    int mantissa = code & 7;
    double magnitude;
    if (exponent == 15 && mantissa == 7) {
        magnitude = NAN;
    } else if (exponent == 0) {
        magnitude = ldexp((double)mantissa, -9);
    } else {
        magnitude = ldexp((double)(8 + mantissa), exponent - 10);
    }
    return sign ? -magnitude : magnitude;
}

/* Nearest E4M3 code of a binary32 value, ties to the even code.  In the
 * binade [2^e, 2^(e+1)), e >= -6, neighbouring values are 2^(e-3) apart;
 * below 2^-6 (the subnormals) they are 2^-9 apart, the spacing of e = -6.
 * With steps = |x| / spacing rounded to an integer r, the code is
 * (e + 7) * 8 + (r - 8): r = 16 carries into the next binade and r < 8
 * gives the subnormal codes.  Magnitudes of 448 and above, infinities
 * included, saturate to 448; NaN gives 0x7f. */
uint8_t oracle_e4m3_from_f32(float x) {
    if (isnan(x)) return 0x7f;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7e;
    int e = -6;
    if (a >= ldexp(1.0, -6)) {
        int exponent;
        frexp(a, &exponent); /* a = f * 2^exponent, f in [0.5, 1) */
        e = exponent - 1;
    }
    const double steps = a / ldexp(1.0, e - 3); /* exact: division by a power of two */
    double r = floor(steps);
    const double remainder = steps - r;
    if (remainder > 0.5 || (remainder == 0.5 && fmod(r, 2.0) == 1.0)) r += 1.0;
    return (uint8_t)(sign | ((e + 7) * 8 + ((int)r - 8)));
}

/* ------------------------------------------------------------------ */
/* Gather: logical token t of sequence s lives in physical block         */
/* block_tables[s][t / B], slot t % B (vLLM PagedAttention & continuous  */
/* batching, "PagedAttention: fixed blocks, non-contiguous physical      */
/* memory": a block table maps each logical block to a physical block,  */
/* logical blocks fill left to right).                                   */
/* ------------------------------------------------------------------ */

/* Copies the n tokens of (sequence s, KV head h) into contiguous binary64
 * rows dst[t][0..head_dim).  Returns ORACLE_BAD_INDEX if a block id used
 * by the sequence is outside the pool. */
static int gather_contiguous(const uint16_t *cache, int dtype, int num_blocks, int num_kv_heads,
                             int block_size, int head_dim, const int32_t *table_row, int n, int h,
                             double *dst) {
    for (int t = 0; t < n; ++t) {
        int32_t physical = table_row[t / block_size];
        int slot = t % block_size;
        if (physical < 0 || physical >= num_blocks) return ORACLE_BAD_INDEX;
        const uint16_t *row =
            cache + (((size_t)physical * num_kv_heads + h) * block_size + slot) * head_dim;
        for (int k = 0; k < head_dim; ++k) dst[(size_t)t * head_dim + k] = widen(row[k], dtype);
    }
    return ORACLE_OK;
}

/* The same gather from a pool of E4M3 codes: each value is read back as
 * code * factor (the pool's scale), exactly, in binary64. */
static int gather_contiguous_e4m3(const uint8_t *cache, double factor, int num_blocks,
                                  int num_kv_heads, int block_size, int head_dim,
                                  const int32_t *table_row, int n, int h, double *dst) {
    for (int t = 0; t < n; ++t) {
        int32_t physical = table_row[t / block_size];
        int slot = t % block_size;
        if (physical < 0 || physical >= num_blocks) return ORACLE_BAD_INDEX;
        const uint8_t *row =
            cache + (((size_t)physical * num_kv_heads + h) * block_size + slot) * head_dim;
        for (int k = 0; k < head_dim; ++k)
            dst[(size_t)t * head_dim + k] = factor * oracle_e4m3_to_f64(row[k]);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Dense attention on the contiguous copy, two passes, binary64.         */
/* PagedAttention keeps the attention maths unchanged and only changes    */
/* storage (vLLM PagedAttention & continuous batching, "PagedAttention";  */
/* the paper's "formula is unchanged", "The kernel page").  Outputs are   */
/* checked "against a contiguous-KV baseline" (PagedAttention and Online  */
/* Inference, "Verification and Experimental Plan", item 1).             */
/*                                                                       */
/* Query head i reads KV head floor(i / g), g = num_q_heads/num_kv_heads  */
/* (grouped-query / multi-query attention, PagedAttention and Online      */
/* Inference section 1; contiguous groups is the plainest mapping).       */
/* An empty sequence (n = 0) yields a zero output row.                    */
/* ------------------------------------------------------------------ */
/* Two-pass dense softmax of the `group` query heads of KV head h of
 * sequence s over its n gathered key / value rows. */
static void attend_group(const uint16_t *q, int dtype, int s, int h, int group, int num_q_heads,
                         int head_dim, int n, const double *keys, const double *values,
                         double *scores, double scale, double *out_group) {
    for (int i = 0; i < group; ++i) {
        const int qh = h * group + i;
        const uint16_t *q_row = q + ((size_t)s * num_q_heads + qh) * head_dim;
        /* pass 1: scaled scores and their maximum */
        double m = -INFINITY;
        for (int t = 0; t < n; ++t) {
            double dot = 0.0;
            for (int k = 0; k < head_dim; ++k)
                dot += widen(q_row[k], dtype) * keys[(size_t)t * head_dim + k];
            scores[t] = scale * dot;
            if (scores[t] > m) m = scores[t];
        }
        /* pass 2: exp(s - max), normaliser and weighted sum of values */
        double denominator = 0.0;
        double *o = out_group + (size_t)i * head_dim;
        for (int k = 0; k < head_dim; ++k) o[k] = 0.0;
        for (int t = 0; t < n; ++t) {
            double p = exp(scores[t] - m);
            denominator += p;
            for (int k = 0; k < head_dim; ++k) o[k] += p * values[(size_t)t * head_dim + k];
        }
        for (int k = 0; k < head_dim; ++k) o[k] /= denominator;
    }
}

/* Pools of 16-bit scalars (fp8 == 0) or of E4M3 codes with scale factors
 * k_factor / v_factor (fp8 == 1). */
static int paged_attention(const uint16_t *q, int dtype, int num_seqs, int num_q_heads,
                           const void *k_cache, const void *v_cache, int fp8, double k_factor,
                           double v_factor, int num_blocks, int num_kv_heads, int block_size,
                           int head_dim, const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *seq_lens, double scale, double *out, int num_threads) {
    if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || block_size <= 0 ||
        head_dim <= 0 || (dtype != 0 && dtype != 1))
        return ORACLE_BAD_ARG;
    const int group = num_q_heads / num_kv_heads;
    int status = ORACLE_OK;
    const long long pairs = (long long)num_seqs * num_kv_heads;
    if (num_threads < 1) num_threads = 1;

#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
    for (long long pair = 0; pair < pairs; ++pair) {
        const int s = (int)(pair / num_kv_heads);
        const int h = (int)(pair % num_kv_heads);
        const int n = seq_lens[s];
        double *out_group = out + ((size_t)s * num_q_heads + (size_t)h * group) * head_dim;
        if (n <= 0) {
            for (size_t e = 0; e < (size_t)group * head_dim; ++e) out_group[e] = 0.0;
            continue;
        }
        if (n > max_blocks_per_seq * block_size) {
#pragma omp atomic write
            status = ORACLE_BAD_INDEX;
            continue;
        }
        double *keys = malloc(sizeof(double) * (size_t)n * head_dim);
        double *values = malloc(sizeof(double) * (size_t)n * head_dim);
        double *scores = malloc(sizeof(double) * (size_t)n);
        if (!keys || !values || !scores) {
            free(keys); free(values); free(scores);
#pragma omp atomic write
            status = ORACLE_NO_MEMORY;
            continue;
        }
        const int32_t *table_row = block_tables + (size_t)s * max_blocks_per_seq;
        int gk, gv;
        if (fp8) {
            gk = gather_contiguous_e4m3(k_cache, k_factor, num_blocks, num_kv_heads, block_size,
                                        head_dim, table_row, n, h, keys);
            gv = gather_contiguous_e4m3(v_cache, v_factor, num_blocks, num_kv_heads, block_size,
                                        head_dim, table_row, n, h, values);
        } else {
            gk = gather_contiguous(k_cache, dtype, num_blocks, num_kv_heads, block_size, head_dim,
                                   table_row, n, h, keys);
            gv = gather_contiguous(v_cache, dtype, num_blocks, num_kv_heads, block_size, head_dim,
                                   table_row, n, h, values);
        }
        if (gk != ORACLE_OK || gv != ORACLE_OK) {
            free(keys); free(values); free(scores);
#pragma omp atomic write
            status = ORACLE_BAD_INDEX;
            continue;
        }
        attend_group(q, dtype, s, h, group, num_q_heads, head_dim, n, keys, values, scores, scale,
                     out_group);
        free(keys); free(values); free(scores);
    }
    return status;
}

int oracle_paged_attention(const uint16_t *q, int dtype, int num_seqs, int num_q_heads,
                           const uint16_t *k_cache, const uint16_t *v_cache, int num_blocks,
                           int num_kv_heads, int block_size, int head_dim,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *seq_lens, double scale, double *out, int num_threads) {
    return paged_attention(q, dtype, num_seqs, num_q_heads, k_cache, v_cache, 0, 1.0, 1.0,
                           num_blocks, num_kv_heads, block_size, head_dim, block_tables,
                           max_blocks_per_seq, seq_lens, scale, out, num_threads);
}

/* The same attention over pools of E4M3 codes: key t of the formula is
 * k_scale * decode(code), value t is v_scale * decode(code). */
int oracle_paged_attention_fp8(const uint16_t *q, int dtype, int num_seqs, int num_q_heads,
                               const uint8_t *k_cache, const uint8_t *v_cache, int num_blocks,
                               int num_kv_heads, int block_size, int head_dim,
                               const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *seq_lens, double scale, float k_scale,
                               float v_scale, double *out, int num_threads) {
    return paged_attention(q, dtype, num_seqs, num_q_heads, k_cache, v_cache, 1, (double)k_scale,
                           (double)v_scale, num_blocks, num_kv_heads, block_size, head_dim,
                           block_tables, max_blocks_per_seq, seq_lens, scale, out, num_threads);
}

/* ------------------------------------------------------------------ */
/* The same attention by the online recurrence of Serving Language      */
/* Models Within a Memory Budget, Eq. (4): for each new block of scores  */
/*     m' = max(m, max_j s_j),  l' = e^(m - m') l + sum_j e^(s_j - m'),   */
/* and the weighted-value accumulator is rescaled by the same factor     */
/* e^(m - m').  Tokens are visited in consecutive chunks of `chunk`      */
/* tokens (any positive size; it need not equal the block size).  This   */
/* exists only to check that the recurrence equals the two-pass result.  */
/* ------------------------------------------------------------------ */
int oracle_online_attention(const uint16_t *q, int dtype, int num_seqs, int num_q_heads,
                            const uint16_t *k_cache, const uint16_t *v_cache, int num_blocks,
                            int num_kv_heads, int block_size, int head_dim,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *seq_lens, double scale, int chunk, double *out) {
    if (chunk <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0)
        return ORACLE_BAD_ARG;
    const int group = num_q_heads / num_kv_heads;
    double *acc = malloc(sizeof(double) * (size_t)head_dim);
    if (!acc) return ORACLE_NO_MEMORY;
    for (int s = 0; s < num_seqs; ++s) {
        const int n = seq_lens[s];
        if (n > max_blocks_per_seq * block_size) { free(acc); return ORACLE_BAD_INDEX; }
        const int32_t *table_row = block_tables + (size_t)s * max_blocks_per_seq;
        for (int qh = 0; qh < num_q_heads; ++qh) {
            const int h = qh / group;
            const uint16_t *q_row = q + ((size_t)s * num_q_heads + qh) * head_dim;
            double m = -INFINITY, l = 0.0;
            for (int k = 0; k < head_dim; ++k) acc[k] = 0.0;
            for (int start = 0; start < n; start += chunk) {
                const int stop = start + chunk < n ? start + chunk : n;
                /* scores of this chunk and their maximum */
                double chunk_max = -INFINITY;
                double *chunk_scores = malloc(sizeof(double) * (size_t)(stop - start));
                if (!chunk_scores) { free(acc); return ORACLE_NO_MEMORY; }
                for (int t = start; t < stop; ++t) {
                    int32_t physical = table_row[t / block_size];
                    if (physical < 0 || physical >= num_blocks) {
                        free(chunk_scores); free(acc); return ORACLE_BAD_INDEX;
                    }
                    const uint16_t *k_row = k_cache + (((size_t)physical * num_kv_heads + h) *
                                                       block_size + t % block_size) * head_dim;
                    double dot = 0.0;
                    for (int k = 0; k < head_dim; ++k)
                        dot += widen(q_row[k], dtype) * widen(k_row[k], dtype);
                    chunk_scores[t - start] = scale * dot;
                    if (chunk_scores[t - start] > chunk_max) chunk_max = chunk_scores[t - start];
                }
                const double m_new = m > chunk_max ? m : chunk_max;
                const double rescale = exp(m - m_new); /* e^(m - m'); 0 when m = -inf */
                l *= rescale;
                for (int k = 0; k < head_dim; ++k) acc[k] *= rescale;
                for (int t = start; t < stop; ++t) {
                    int32_t physical = table_row[t / block_size];
                    const uint16_t *v_row = v_cache + (((size_t)physical * num_kv_heads + h) *
                                                       block_size + t % block_size) * head_dim;
                    double p = exp(chunk_scores[t - start] - m_new);
                    l += p;
                    for (int k = 0; k < head_dim; ++k) acc[k] += p * widen(v_row[k], dtype);
                }
                m = m_new;
                free(chunk_scores);
            }
            double *o = out + ((size_t)s * num_q_heads + qh) * head_dim;
            for (int k = 0; k < head_dim; ++k) o[k] = n > 0 ? acc[k] / l : 0.0;
        }
    }
    free(acc);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Per-partition softmax statistics for the split over the sequence.    */
/* Partition p of sequence s covers tokens [p*P, min((p+1)*P, n)).  For  */
/* each (s, query head, p):                                              */
/*     m_p = max of the partition's scaled scores,                        */
/*     l_p = sum of e^(s_t - m_p),   acc_p = sum of e^(s_t - m_p) v_t.    */
/* Partitions past the end of a sequence get m = -inf, l = 0, acc = 0.    */
/* Layout: m, l [S][H_q][num_partitions]; acc [S][H_q][num_partitions][d]  */
/* ------------------------------------------------------------------ */
int oracle_partition_stats(const uint16_t *q, int dtype, int num_seqs, int num_q_heads,
                           const uint16_t *k_cache, const uint16_t *v_cache, int num_blocks,
                           int num_kv_heads, int block_size, int head_dim,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *seq_lens, double scale, int partition_size,
                           int num_partitions, double *m_out, double *l_out, double *acc_out) {
    if (partition_size <= 0 || num_partitions <= 0 || num_kv_heads <= 0 ||
        num_q_heads % num_kv_heads != 0)
        return ORACLE_BAD_ARG;
    const int group = num_q_heads / num_kv_heads;
    for (int s = 0; s < num_seqs; ++s) {
        const int n = seq_lens[s];
        if (n > max_blocks_per_seq * block_size || n > partition_size * num_partitions)
            return ORACLE_BAD_INDEX;
        const int32_t *table_row = block_tables + (size_t)s * max_blocks_per_seq;
        for (int qh = 0; qh < num_q_heads; ++qh) {
            const int h = qh / group;
            const uint16_t *q_row = q + ((size_t)s * num_q_heads + qh) * head_dim;
            for (int p = 0; p < num_partitions; ++p) {
                const size_t idx = ((size_t)s * num_q_heads + qh) * num_partitions + p;
                double *acc = acc_out + idx * head_dim;
                const int start = p * partition_size;
                const int stop = start + partition_size < n ? start + partition_size : n;
                double m = -INFINITY, l = 0.0;
                for (int k = 0; k < head_dim; ++k) acc[k] = 0.0;
                if (start < stop) {
                    double *scores = malloc(sizeof(double) * (size_t)(stop - start));
                    if (!scores) return ORACLE_NO_MEMORY;
                    for (int t = start; t < stop; ++t) {
                        int32_t physical = table_row[t / block_size];
                        if (physical < 0 || physical >= num_blocks) { free(scores); return ORACLE_BAD_INDEX; }
                        const uint16_t *k_row = k_cache + (((size_t)physical * num_kv_heads + h) *
                                                           block_size + t % block_size) * head_dim;
                        double dot = 0.0;
                        for (int k = 0; k < head_dim; ++k)
                            dot += widen(q_row[k], dtype) * widen(k_row[k], dtype);
                        scores[t - start] = scale * dot;
                        if (scores[t - start] > m) m = scores[t - start];
                    }
                    for (int t = start; t < stop; ++t) {
                        int32_t physical = table_row[t / block_size];
                        const uint16_t *v_row = v_cache + (((size_t)physical * num_kv_heads + h) *
                                                           block_size + t % block_size) * head_dim;
                        double w = exp(scores[t - start] - m);
                        l += w;
                        for (int k = 0; k < head_dim; ++k) acc[k] += w * widen(v_row[k], dtype);
                    }
                    free(scores);
                }
                m_out[idx] = m;
                l_out[idx] = l;
            }
        }
    }
    return ORACLE_OK;
}

/* Merge of partition statistics: Eq. (4) of Serving Language Models Within
 * a Memory Budget applied with each partition as one "block":
 *     M = max_p m_p,  out = sum_p e^(m_p - M) acc_p / sum_p e^(m_p - M) l_p.
 * rows = number of (sequence, query head) rows; all-empty rows give 0. */
int oracle_merge_partitions(const double *m_in, const double *l_in, const double *acc_in,
                            long long rows, int num_partitions, int head_dim, double *out) {
    for (long long r = 0; r < rows; ++r) {
        const double *m = m_in + r * num_partitions;
        const double *l = l_in + r * num_partitions;
        double big = -INFINITY;
        for (int p = 0; p < num_partitions; ++p) if (m[p] > big) big = m[p];
        double *o = out + r * head_dim;
        for (int k = 0; k < head_dim; ++k) o[k] = 0.0;
        if (big == -INFINITY) continue;
        double denominator = 0.0;
        for (int p = 0; p < num_partitions; ++p) {
            if (m[p] == -INFINITY) continue;
            double w = exp(m[p] - big);
            denominator += w * l[p];
            const double *acc = acc_in + ((size_t)r * num_partitions + p) * head_dim;
            for (int k = 0; k < head_dim; ++k) o[k] += w * acc[k];
        }
        for (int k = 0; k < head_dim; ++k) o[k] /= denominator;
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* KV write through a slot mapping: token t's key and value rows, one per */
/* KV head, go to slot slot_mapping[t] = physical_block * B + offset.    */
/* Decode writes the next token into the spare slot of the last block    */
/* (vLLM PagedAttention & continuous batching, "PagedAttention", the      */
/* seven-token example).  A negative slot marks a padding token and is    */
/* skipped; a slot past the pool is skipped and reported.                */
/* k, v : [num_tokens][num_kv_heads][head_dim]                            */
/* ------------------------------------------------------------------ */
int oracle_kv_write(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping,
                    int num_tokens, uint16_t *k_cache, uint16_t *v_cache, int num_blocks,
                    int num_kv_heads, int block_size, int head_dim) {
    int status = ORACLE_OK;
    for (int t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) { status = ORACLE_BAD_INDEX; continue; }
        const int64_t physical = slot / block_size;
        const int64_t offset = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            const size_t src = ((size_t)t * num_kv_heads + h) * head_dim;
            const size_t dst = (((size_t)physical * num_kv_heads + h) * block_size + offset) * head_dim;
            for (int e = 0; e < head_dim; ++e) {
                k_cache[dst + e] = k[src + e];
                v_cache[dst + e] = v[src + e];
            }
        }
    }
    return status;
}

/* The same slot write into pools of E4M3 codes: element x of a key row is
 * stored as E4M3(x / k_scale), the quotient taken in binary32 (x is exact
 * in binary32), and values likewise with v_scale. */
int oracle_kv_write_fp8(const uint16_t *k, const uint16_t *v, int dtype,
                        const int64_t *slot_mapping, int num_tokens, uint8_t *k_cache,
                        uint8_t *v_cache, int num_blocks, int num_kv_heads, int block_size,
                        int head_dim, float k_scale, float v_scale) {
    if (dtype != 0 && dtype != 1) return ORACLE_BAD_ARG;
    int status = ORACLE_OK;
    for (int t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) { status = ORACLE_BAD_INDEX; continue; }
        const int64_t physical = slot / block_size;
        const int64_t offset = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            const size_t src = ((size_t)t * num_kv_heads + h) * head_dim;
            const size_t dst = (((size_t)physical * num_kv_heads + h) * block_size + offset) * head_dim;
            for (int e = 0; e < head_dim; ++e) {
                const float kx = (float)widen(k[src + e], dtype);
                const float vx = (float)widen(v[src + e], dtype);
                const float k_quotient = kx / k_scale;
                const float v_quotient = vx / v_scale;
                k_cache[dst + e] = oracle_e4m3_from_f32(k_quotient);
                v_cache[dst + e] = oracle_e4m3_from_f32(v_quotient);
            }
        }
    }
    return status;
}

/* ------------------------------------------------------------------ */
/* Copy-on-write block copy: for each (src, dst) pair, in order, the      */
/* whole physical block (every KV head, every slot, filled or not) of     */
/* both caches is copied from src to dst (vLLM PagedAttention &           */
/* continuous batching, "Sharing with reference counts and copy-on-write": */
/* the engine allocates a new block and copies that one block).           */
/* pairs : [num_pairs][2] int64                                           */
/* ------------------------------------------------------------------ */
int oracle_copy_blocks(uint16_t *k_cache, uint16_t *v_cache, int num_blocks, int num_kv_heads,
                       int block_size, int head_dim, const int64_t *pairs, int num_pairs) {
    int status = ORACLE_OK;
    const size_t block_elems = (size_t)num_kv_heads * block_size * head_dim;
    for (int i = 0; i < num_pairs; ++i) {
        const int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            status = ORACLE_BAD_INDEX;
            continue;
        }
        memmove(k_cache + (size_t)dst * block_elems, k_cache + (size_t)src * block_elems,
                block_elems * sizeof(uint16_t));
        memmove(v_cache + (size_t)dst * block_elems, v_cache + (size_t)src * block_elems,
                block_elems * sizeof(uint16_t));
    }
    return status;
}

/* ------------------------------------------------------------------ */
/* Paged prefill attention: the prompt phase runs many query tokens of a  */
/* sequence at once (vLLM PagedAttention & continuous batching, "Prompt  */
/* phase, decode phase": prefill runs the known prompt as matrix-matrix  */
/* work).  Sequence s holds n = seq_lens[s] tokens in its blocks, the    */
/* last q_len = cu_q[s+1] - cu_q[s] of them being this call's queries,   */
/* so query i sits at position ctx + i, ctx = n - q_len (an earlier part */
/* of the prompt, or a shared prefix, already cached).  Causal attention: */
/* query i attends to positions 0 .. ctx + i.  Dense two-pass softmax on  */
/* the contiguous gathered copy, binary64.                                */
/* q, out : [total query tokens][num_q_heads][head_dim]                   */
/* ------------------------------------------------------------------ */
int oracle_paged_prefill(const uint16_t *q, const int32_t *cu_q, int dtype, int num_seqs,
                         int num_q_heads, const uint16_t *k_cache, const uint16_t *v_cache,
                         int num_blocks, int num_kv_heads, int block_size, int head_dim,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *seq_lens, double scale, double *out, int num_threads) {
    if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || block_size <= 0 ||
        head_dim <= 0 || (dtype != 0 && dtype != 1))
        return ORACLE_BAD_ARG;
    const int group = num_q_heads / num_kv_heads;
    int status = ORACLE_OK;
    const long long pairs = (long long)num_seqs * num_kv_heads;
    if (num_threads < 1) num_threads = 1;

#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
    for (long long pair = 0; pair < pairs; ++pair) {
        const int s = (int)(pair / num_kv_heads);
        const int h = (int)(pair % num_kv_heads);
        const int n = seq_lens[s];
        const int q_len = cu_q[s + 1] - cu_q[s];
        const int ctx = n - q_len;
        if (q_len < 0 || ctx < 0 || n > max_blocks_per_seq * block_size) {
#pragma omp atomic write
            status = ORACLE_BAD_INDEX;
            continue;
        }
        if (q_len == 0) continue;
        double *keys = malloc(sizeof(double) * (size_t)n * head_dim);
        double *values = malloc(sizeof(double) * (size_t)n * head_dim);
        double *scores = malloc(sizeof(double) * (size_t)n);
        if (!keys || !values || !scores) {
            free(keys); free(values); free(scores);
#pragma omp atomic write
            status = ORACLE_NO_MEMORY;
            continue;
        }
        const int32_t *table_row = block_tables + (size_t)s * max_blocks_per_seq;
        int gk = gather_contiguous(k_cache, dtype, num_blocks, num_kv_heads, block_size, head_dim,
                                   table_row, n, h, keys);
        int gv = gather_contiguous(v_cache, dtype, num_blocks, num_kv_heads, block_size, head_dim,
                                   table_row, n, h, values);
        if (gk != ORACLE_OK || gv != ORACLE_OK) {
            free(keys); free(values); free(scores);
#pragma omp atomic write
            status = ORACLE_BAD_INDEX;
            continue;
        }
        for (int i = 0; i < q_len; ++i) {
            const int visible = ctx + i + 1; /* causal: positions 0 .. ctx + i */
            for (int j = 0; j < group; ++j) {
                const int qh = h * group + j;
                const size_t row = ((size_t)(cu_q[s] + i) * num_q_heads + qh) * head_dim;
                double m = -INFINITY;
                for (int t = 0; t < visible; ++t) {
                    double dot = 0.0;
                    for (int k = 0; k < head_dim; ++k)
                        dot += widen(q[row + k], dtype) * keys[(size_t)t * head_dim + k];
                    scores[t] = scale * dot;
                    if (scores[t] > m) m = scores[t];
                }
                double denominator = 0.0;
                double *o = out + row;
                for (int k = 0; k < head_dim; ++k) o[k] = 0.0;
                for (int t = 0; t < visible; ++t) {
                    double p = exp(scores[t] - m);
                    denominator += p;
                    for (int k = 0; k < head_dim; ++k) o[k] += p * values[(size_t)t * head_dim + k];
                }
                for (int k = 0; k < head_dim; ++k) o[k] /= denominator;
            }
        }
        free(keys); free(values); free(scores);
    }
    return status;
}

/* ------------------------------------------------------------------ */
/* Block transfer between two pools (swap out to, or in from, a second   */
/* pool in host memory: vLLM PagedAttention & continuous batching,        */
/* "Preemption when blocks run out", Swap).  For each (src, dst) pair, in */
/* order, the whole block src of the source pools is copied to block dst  */
/* of the destination pools.                                              */
/* ------------------------------------------------------------------ */
int oracle_transfer_blocks(const uint16_t *src_k, const uint16_t *src_v, int src_num_blocks,
                           uint16_t *dst_k, uint16_t *dst_v, int dst_num_blocks,
                           int num_kv_heads, int block_size, int head_dim, const int64_t *pairs,
                           int num_pairs) {
    int status = ORACLE_OK;
    const size_t block_elems = (size_t)num_kv_heads * block_size * head_dim;
    for (int i = 0; i < num_pairs; ++i) {
        const int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) {
            status = ORACLE_BAD_INDEX;
            continue;
        }
        memcpy(dst_k + (size_t)dst * block_elems, src_k + (size_t)src * block_elems,
               block_elems * sizeof(uint16_t));
        memcpy(dst_v + (size_t)dst * block_elems, src_v + (size_t)src * block_elems,
               block_elems * sizeof(uint16_t));
    }
    return status;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
