/*
 * oracle.c -- plain, slow, single-threaded fp64 CPU oracle for the paged-attention
 * decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the benchmark's
 * CPU-baseline leg are the only callers.  The CUDA path never links, loads or calls
 * this file, and this file includes nothing from the CUDA path.
 *
 * Sources (web pages, cited by title and section):
 *   [TALK]  "vLLM Project Update" (Bay.Area.AI talk transcript, Zhuohan Li and
 *           Woosuk Kwon): the opening part on PagedAttention ("a new attention
 *           algorithm that operates on blocks of KV cache", KV cache managed like
 *           virtual memory) and the part on the new PagedAttention V2 kernel
 *           (each sequence partitioned into smaller pieces spread over SMs,
 *           "similar to flash decoding").
 *   [HN]    "vLLM: Easy, Fast, and Cheap LLM Serving with PagedAttention" (Hacker
 *           News thread): the quoted blog paragraph on the KV cache (1.7 GB per
 *           LLaMA-13B sequence) and the replies that call PagedAttention and
 *           FlashAttention orthogonal ways to compute exact attention.
 *   [PR]    "[core] Multi Step Scheduling #7000": the review snippet that advances
 *           seq_lens, slot_mapping and block_tables between decode steps, and the
 *           launch command using --use-v2-block-manager.
 *
 * Readings taken where the pages are silent (each function repeats its own):
 *   - KV pool layout: key and value pools are separate arrays
 *     [num_blocks][num_kv_heads][block_size][head_size] of 16-bit elements.
 *   - Query head h reads kv head h / (num_q_heads / num_kv_heads).
 *   - context_lens[s] counts the new token, which was scattered before the decode.
 *   - context_len == 0 gives an all-zero output row.
 *   - slot_mapping < 0 marks a padding token: nothing is written.
 *   - V2 partitions a sequence into runs of partition_size tokens; each run keeps
 *     (m_p, l_p, o_p) with o_p normalised; runs are merged by log-sum-exp.
 *   - scale is an fp32 value; the oracle widens it exactly to double.
 *   - Output rounding to fp16/bf16 is round-to-nearest-even from the double result.
 *
 * Built with -ffp-contract=off so that x86 and Arm hosts produce the same doubles.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F16 0
#define OR_BF16 1

/* ------------------------------------------------------------------------- */
/* 16-bit float formats <-> double, written from the IEEE-754 field layouts.   */
/* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits.                   */
/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits.                   */
/* ------------------------------------------------------------------------- */

static double bits_to_double(uint16_t b, int frac_bits, int exp_bits) {
    int bias = (1 << (exp_bits - 1)) - 1;
    int sign = (b >> 15) & 1;
    int e = (b >> frac_bits) & ((1 << exp_bits) - 1);
    int f = b & ((1 << frac_bits) - 1);
    double v;
    if (e == 0) {
        /* zero or subnormal: f * 2^(1 - bias - frac_bits) */
        v = ldexp((double)f, 1 - bias - frac_bits);
    } else if (e == (1 << exp_bits) - 1) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(f | (1 << frac_bits)), e - bias - frac_bits);
    }
    return sign ? -v : v;
}

/* Round a double to the nearest representable value of the format, ties to even,
 * and return its bit pattern.  Works in exact integer arithmetic on the scaled
 * significand: every intermediate below is exact in double. */
static uint16_t double_to_bits(double x, int frac_bits, int exp_bits) {
    int bias = (1 << (exp_bits - 1)) - 1;
    int emax = bias;               /* largest unbiased exponent of a finite value */
    int emin = 1 - bias;           /* smallest unbiased exponent of a normal value */
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    uint16_t exp_all = (uint16_t)(((1 << exp_bits) - 1) << frac_bits);
    if (isnan(x)) return (uint16_t)(sign | exp_all | (1 << (frac_bits - 1)));
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | exp_all);
    int e2;
    (void)frexp(a, &e2);           /* a = f * 2^e2, f in [0.5, 1) */
    int k = e2 - 1;                /* a in [2^k, 2^(k+1)) */
    if (k > emax + 1) return (uint16_t)(sign | exp_all);
    if (k < emin) k = emin;        /* subnormal range shares the quantum of 2^emin */
    double n = ldexp(a, frac_bits - k);   /* significand in units of the quantum */
    double r = nearbyint(n);              /* default rounding mode: ties to even */
    double one = ldexp(1.0, frac_bits);
    if (r >= 2.0 * one) {                 /* rounded up into the next binade */
        r = one;
        k += 1;
    }
    if (k > emax) return (uint16_t)(sign | exp_all);
    if (r < one) {                        /* subnormal (only possible when k == emin) */
        return (uint16_t)(sign | (uint16_t)r);
    }
    uint16_t biased = (uint16_t)(k + bias);
    return (uint16_t)(sign | (uint16_t)(biased << frac_bits) | (uint16_t)(r - one));
}

double or_f16_to_f64(uint16_t b) { return bits_to_double(b, 10, 5); }
double or_bf16_to_f64(uint16_t b) { return bits_to_double(b, 7, 8); }
uint16_t or_f64_to_f16(double x) { return double_to_bits(x, 10, 5); }
uint16_t or_f64_to_bf16(double x) { return double_to_bits(x, 7, 8); }

/* ------------------------------------------------------------------------- */
/* fp8 E4M3 (OCP "E4M3FN"): 1 sign, 4 exponent (bias 7), 3 fraction bits; no     */
/* infinities; S.1111.111 is NaN; largest finite 448.  Used for the fp8 KV cache   */
/* the "vLLM Project Update" talk lists among the supported quantisation methods.  */
/* ------------------------------------------------------------------------- */
double or_e4m3_to_f64(uint8_t b) {
    int sign = (b >> 7) & 1, e = (b >> 3) & 15, f = b & 7;
    double v;
    if (e == 15 && f == 7) return NAN;
    if (e == 0) v = ldexp((double)f, -9);                 /* subnormal: f * 2^(1-7-3) */
    else v = ldexp((double)(f | 8), e - 10);              /* (8+f) * 2^(e-7-3) */
    return sign ? -v : v;
}

/* Round to E4M3, nearest with ties to even; finite values beyond 448 saturate to
 * +-448 (the fp8 KV cache stores finite numbers only); NaN stays NaN. */
uint8_t or_f64_to_e4m3(double x) {
    uint8_t sign = signbit(x) ? 0x80 : 0;
    if (isnan(x)) return (uint8_t)(sign | 0x7F);
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);        /* 448 = 1.75 * 2^8 */
    int e2;
    (void)frexp(a, &e2);
    int k = e2 - 1;                                       /* a in [2^k, 2^(k+1)) */
    if (k < -6) k = -6;                                   /* subnormals share 2^-6's quantum */
    double n = ldexp(a, 3 - k);
    double r = nearbyint(n);
    if (r >= 16.0) { r = 8.0; k += 1; }
    if (k > 8 || (k == 8 && r > 14.0)) return (uint8_t)(sign | 0x7E);   /* rounds past 448 */
    if (r < 8.0) return (uint8_t)(sign | (uint8_t)r);     /* subnormal (k == -6) */
    return (uint8_t)(sign | (uint8_t)((k + 7) << 3) | (uint8_t)(r - 8.0));
}

void or_e4m3_widen_array(const uint8_t* in, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_e4m3_to_f64(in[i]);
}

void or_e4m3_round_array(const double* in, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_f64_to_e4m3(in[i]);
}

static double widen(uint16_t b, int dtype) {
    return dtype == OR_BF16 ? or_bf16_to_f64(b) : or_f16_to_f64(b);
}

/* Vector forms, for the tests' convenience. */
void or_widen_array(const uint16_t* in, double* out, int64_t n, int32_t dtype) {
    for (int64_t i = 0; i < n; ++i) out[i] = widen(in[i], dtype);
}

void or_round_array(const double* in, uint16_t* out, int64_t n, int32_t dtype) {
    for (int64_t i = 0; i < n; ++i)
        out[i] = dtype == OR_BF16 ? or_f64_to_bf16(in[i]) : or_f64_to_f16(in[i]);
}

/* ------------------------------------------------------------------------- */
/* reshape_and_cache: scatter each new token's K and V rows into the pools.    */
/* [PR] slot_mapping names, per new token, the flat slot                       */
/* block * block_size + offset it occupies; [TALK] the pool is a set of        */
/* fixed-size blocks.  Reading: slot < 0 is a padding token (skipped); a slot  */
/* at or beyond num_blocks * block_size is an error and is skipped too.        */
/* Returns the number of skipped out-of-range slots.                          */
/* ------------------------------------------------------------------------- */
int32_t or_reshape_and_cache(const uint16_t* key, const uint16_t* value,
                             uint16_t* key_cache, uint16_t* value_cache,
                             const int32_t* slot_mapping, int32_t num_tokens,
                             int32_t num_kv_heads, int32_t head_size,
                             int32_t block_size, int32_t num_blocks) {
    int32_t bad = 0;
    for (int32_t i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) { ++bad; continue; }
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            for (int32_t d = 0; d < head_size; ++d) {
                int64_t src = ((int64_t)i * num_kv_heads + h) * head_size + d;
                int64_t dst = ((block * num_kv_heads + h) * block_size + offset) * head_size + d;
                key_cache[dst] = key[src];
                value_cache[dst] = value[src];
            }
        }
    }
    return bad;
}

/* ------------------------------------------------------------------------- */
/* Paged decode attention.                                                    */
/* ------------------------------------------------------------------------- */

typedef struct {
    const uint16_t* q;
    const uint16_t* k_cache;
    const uint16_t* v_cache;
    const int32_t* block_tables;
    int32_t max_blocks_per_seq;
    const int32_t* context_lens;
    int32_t num_seqs, num_q_heads, num_kv_heads, head_size, block_size, num_blocks;
    double scale;
    int32_t dtype;
} decode_args;

/* Element d of the K (or V) row of token t of sequence s for kv head kvh, found by
 * going through the block table: logical block t / block_size, row t % block_size.
 * Returns 0 and sets *bad when the table entry is outside the pool. */
static double cache_at(const decode_args* a, const uint16_t* cache, int32_t s,
                       int32_t kvh, int32_t t, int32_t d, int* bad) {
    int32_t logical = t / a->block_size;
    int32_t row = t % a->block_size;
    if (logical >= a->max_blocks_per_seq) { *bad = 1; return 0.0; }
    int32_t phys = a->block_tables[(int64_t)s * a->max_blocks_per_seq + logical];
    if (phys < 0 || phys >= a->num_blocks) { *bad = 1; return 0.0; }
    int64_t idx = (((int64_t)phys * a->num_kv_heads + kvh) * a->block_size + row) * a->head_size + d;
    return widen(cache[idx], a->dtype);
}

/* Scaled dot products l_t = scale * sum_d q_d k_t,d for tokens [t0, t1), q_d being
 * element d of the query row `qrow` of query head h. */
static void logits_range(const decode_args* a, const uint16_t* qrow, int32_t s, int32_t h,
                         int32_t t0, int32_t t1, double* logit, int* bad) {
    int32_t group = a->num_q_heads / a->num_kv_heads;
    int32_t kvh = h / group;
    for (int32_t t = t0; t < t1; ++t) {
        double acc = 0.0;
        for (int32_t d = 0; d < a->head_size; ++d)
            acc += widen(qrow[d], a->dtype) * cache_at(a, a->k_cache, s, kvh, t, d, bad);
        logit[t - t0] = a->scale * acc;
    }
}

/* Softmax-weighted sum of V over tokens [t0, t1) of sequence s for query head h, whose
 * query row is `qrow`:
 *   m = max l_t,  p_t = exp(l_t - m),  l = sum p_t,  o = sum p_t v_t / l.
 * Writes o (head_size values) and returns m and l through the pointers. */
static void attend_range(const decode_args* a, const uint16_t* qrow, int32_t s, int32_t h,
                         int32_t t0, int32_t t1, double* o, double* m_out, double* l_out,
                         double* scratch, int* bad) {
    int32_t group = a->num_q_heads / a->num_kv_heads;
    int32_t kvh = h / group;
    int32_t n = t1 - t0;
    logits_range(a, qrow, s, h, t0, t1, scratch, bad);
    double m = -INFINITY;
    for (int32_t i = 0; i < n; ++i) if (scratch[i] > m) m = scratch[i];
    double l = 0.0;
    for (int32_t i = 0; i < n; ++i) { scratch[i] = exp(scratch[i] - m); l += scratch[i]; }
    for (int32_t d = 0; d < a->head_size; ++d) {
        double acc = 0.0;
        for (int32_t i = 0; i < n; ++i)
            acc += scratch[i] * cache_at(a, a->v_cache, s, kvh, t0 + i, d, bad);
        o[d] = acc / l;
    }
    *m_out = m;
    *l_out = l;
}

static int32_t check_shapes(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                            int32_t block_size) {
    if (num_q_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0) return -2;
    if (num_q_heads % num_kv_heads != 0) return -2;
    return 0;
}

/* V1 (one pass over the whole context of each sequence):
 * out[s][h][:] = softmax(scale * q K^T) V over tokens 0..context_lens[s]-1, gathered
 * through the block table ([TALK], PagedAttention; [HN], exact attention).
 * `only` (optional, [num_seqs * num_q_heads] of 0/1) restricts the work to the
 * marked (sequence, head) rows; other rows of `out` are left untouched.
 * Returns 0, -1 if a block-table entry was out of range, -2 on bad shapes. */
int32_t or_paged_decode_v1(double* out, const uint16_t* q, const uint16_t* k_cache,
                           const uint16_t* v_cache, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens,
                           int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_size, int32_t block_size, int32_t num_blocks,
                           float scale, int32_t dtype, const uint8_t* only) {
    int32_t rc = check_shapes(num_q_heads, num_kv_heads, head_size, block_size);
    if (rc) return rc;
    decode_args a = {q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                     num_seqs, num_q_heads, num_kv_heads, head_size, block_size, num_blocks,
                     (double)scale, dtype};
    int bad = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        int32_t L = context_lens[s];
        double* scratch = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        for (int32_t h = 0; h < num_q_heads; ++h) {
            if (only && !only[(int64_t)s * num_q_heads + h]) continue;
            double* o = out + ((int64_t)s * num_q_heads + h) * head_size;
            if (L <= 0) {                       /* reading: empty context -> zeros */
                for (int32_t d = 0; d < head_size; ++d) o[d] = 0.0;
                continue;
            }
            const uint16_t* qrow = q + ((int64_t)s * num_q_heads + h) * head_size;
            double m, l;
            attend_range(&a, qrow, s, h, 0, L, o, &m, &l, scratch, &bad);
        }
        free(scratch);
    }
    return bad ? -1 : 0;
}

/* V2 ([TALK], PagedAttention V2, "similar to flash decoding"): the context of each
 * sequence is cut into partitions of partition_size tokens,
 *   [p * P, min((p + 1) * P, L)),
 * each partition p yields (m_p, l_p, o_p) as in attend_range, and the partitions are
 * merged by a log-sum-exp reduction:
 *   M = max_p m_p,  w_p = l_p * exp(m_p - M),  out = sum_p w_p o_p / sum_p w_p.
 * Same arguments and return codes as V1, plus partition_size (> 0). */
int32_t or_paged_decode_v2(double* out, const uint16_t* q, const uint16_t* k_cache,
                           const uint16_t* v_cache, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens,
                           int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_size, int32_t block_size, int32_t num_blocks,
                           float scale, int32_t dtype, const uint8_t* only,
                           int32_t partition_size) {
    int32_t rc = check_shapes(num_q_heads, num_kv_heads, head_size, block_size);
    if (rc) return rc;
    if (partition_size <= 0) return -2;
    decode_args a = {q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                     num_seqs, num_q_heads, num_kv_heads, head_size, block_size, num_blocks,
                     (double)scale, dtype};
    int bad = 0;
    double* scratch = (double*)malloc(sizeof(double) * (size_t)partition_size);
    for (int32_t s = 0; s < num_seqs; ++s) {
        int32_t L = context_lens[s];
        int32_t np = L > 0 ? (L + partition_size - 1) / partition_size : 0;
        double* mp = (double*)malloc(sizeof(double) * (size_t)(np > 0 ? np : 1));
        double* lp = (double*)malloc(sizeof(double) * (size_t)(np > 0 ? np : 1));
        double* op = (double*)malloc(sizeof(double) * (size_t)(np > 0 ? np : 1) * (size_t)head_size);
        for (int32_t h = 0; h < num_q_heads; ++h) {
            if (only && !only[(int64_t)s * num_q_heads + h]) continue;
            double* o = out + ((int64_t)s * num_q_heads + h) * head_size;
            if (np == 0) {
                for (int32_t d = 0; d < head_size; ++d) o[d] = 0.0;
                continue;
            }
            const uint16_t* qrow = q + ((int64_t)s * num_q_heads + h) * head_size;
            for (int32_t p = 0; p < np; ++p) {
                int32_t t0 = p * partition_size;
                int32_t t1 = t0 + partition_size < L ? t0 + partition_size : L;
                attend_range(&a, qrow, s, h, t0, t1, op + (int64_t)p * head_size, &mp[p], &lp[p],
                             scratch, &bad);
            }
            double M = -INFINITY;
            for (int32_t p = 0; p < np; ++p) if (mp[p] > M) M = mp[p];
            double wsum = 0.0;
            for (int32_t p = 0; p < np; ++p) wsum += lp[p] * exp(mp[p] - M);
            for (int32_t d = 0; d < head_size; ++d) {
                double acc = 0.0;
                for (int32_t p = 0; p < np; ++p)
                    acc += lp[p] * exp(mp[p] - M) * op[(int64_t)p * head_size + d];
                o[d] = acc / wsum;
            }
        }
        free(mp);
        free(lp);
        free(op);
    }
    free(scratch);
    return bad ? -1 : 0;
}

/* Multi-query decode ([TALK]: kernels for several query tokens per sequence, used to
 * verify speculative tokens).  Reading: every sequence brings the same number q_len of
 * new tokens, already scattered, and context_lens[s] counts all of them; new token j
 * (0-based) sits at position L - q_len + j and attends causally to tokens
 * t < L - q_len + j + 1.  query / out are [num_seqs][q_len][num_q_heads][head_size].  A
 * query row with no token to attend to (L < q_len - j) is a zero row. */
int32_t or_paged_decode_mq(double* out, const uint16_t* q, const uint16_t* k_cache,
                           const uint16_t* v_cache, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens,
                           int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                           int32_t num_blocks, float scale, int32_t dtype) {
    int32_t rc = check_shapes(num_q_heads, num_kv_heads, head_size, block_size);
    if (rc) return rc;
    if (q_len <= 0) return -2;
    decode_args a = {q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                     num_seqs, num_q_heads, num_kv_heads, head_size, block_size, num_blocks,
                     (double)scale, dtype};
    int bad = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        int32_t L = context_lens[s];
        double* scratch = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        for (int32_t j = 0; j < q_len; ++j) {
            int32_t limit = L - q_len + j + 1;                  /* tokens this row sees */
            for (int32_t h = 0; h < num_q_heads; ++h) {
                double* o = out + (((int64_t)s * q_len + j) * num_q_heads + h) * head_size;
                if (limit <= 0) {
                    for (int32_t d = 0; d < head_size; ++d) o[d] = 0.0;
                    continue;
                }
                /* the query row of new token j, head h */
                const uint16_t* qrow = q + (((int64_t)s * q_len + j) * num_q_heads + h) * head_size;
                double m, l;
                attend_range(&a, qrow, s, h, 0, limit, o, &m, &l, scratch, &bad);
            }
        }
        free(scratch);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* fp8 KV cache.  Readings: per-tensor scales k_scale, v_scale (> 0); a cached      */
/* element stores e4m3(x * inv) with inv = the fp32 reciprocal of the scale,       */
/* correctly rounded, and x * inv rounded to fp32 first (one fp32 multiply, then   */
/* rounding to E4M3, ties to even, saturating at 448); it reads back as            */
/* decode(e4m3) * scale.  Queries and outputs stay 16-bit.                         */
/* ------------------------------------------------------------------------- */
static uint8_t quantize_e4m3(uint16_t x16, int dtype, float inv) {
    float xf = (float)widen(x16, dtype);        /* exact */
    float prod = xf * inv;                       /* fp32 product, correctly rounded */
    return or_f64_to_e4m3((double)prod);
}

int32_t or_reshape_and_cache_fp8(const uint16_t* key, const uint16_t* value, uint8_t* key_cache,
                                 uint8_t* value_cache, const int32_t* slot_mapping,
                                 int32_t num_tokens, int32_t num_kv_heads, int32_t head_size,
                                 int32_t block_size, int32_t num_blocks, int32_t dtype,
                                 float k_scale, float v_scale) {
    float kinv = 1.0f / k_scale, vinv = 1.0f / v_scale;
    int32_t bad = 0;
    for (int32_t i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) { ++bad; continue; }
        int64_t block = slot / block_size, offset = slot % block_size;
        for (int32_t h = 0; h < num_kv_heads; ++h)
            for (int32_t d = 0; d < head_size; ++d) {
                int64_t src = ((int64_t)i * num_kv_heads + h) * head_size + d;
                int64_t dst = ((block * num_kv_heads + h) * block_size + offset) * head_size + d;
                key_cache[dst] = quantize_e4m3(key[src], dtype, kinv);
                value_cache[dst] = quantize_e4m3(value[src], dtype, vinv);
            }
    }
    return bad;
}

/* Offset of the row of token t (sequence s, kv head kvh) in a pool laid out
 * [num_blocks][num_kv_heads][block_size][head_size], found through the block table; -1
 * (and *bad set) when t's logical block lies past the sequence's table row or the entry
 * lies outside the pool.  Such a token reads as zeros, the same reading as cache_at. */
static int64_t pool_row(const int32_t* block_tables, int32_t max_blocks_per_seq,
                        int32_t num_kv_heads, int32_t block_size, int32_t head_size,
                        int32_t num_blocks, int32_t s, int32_t kvh, int32_t t, int* bad) {
    int32_t logical = t / block_size;
    if (logical >= max_blocks_per_seq) { *bad = 1; return -1; }
    int32_t phys = block_tables[(int64_t)s * max_blocks_per_seq + logical];
    if (phys < 0 || phys >= num_blocks) { *bad = 1; return -1; }
    return (((int64_t)phys * num_kv_heads + kvh) * block_size + t % block_size) * head_size;
}

/* Decode over an fp8 cache: the plain definition with k_t = decode(K8) * k_scale and
 * v_t = decode(V8) * v_scale, everything else as or_paged_decode_v1 (a token whose block
 * the table does not give reads as zeros: logit 0, no V contribution; return -1). */
int32_t or_paged_decode_fp8(double* out, const uint16_t* q, const uint8_t* k_cache,
                            const uint8_t* v_cache, const int32_t* block_tables,
                            int32_t max_blocks_per_seq, const int32_t* context_lens,
                            int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                            int32_t head_size, int32_t block_size, int32_t num_blocks, float scale,
                            float k_scale, float v_scale, int32_t dtype, const uint8_t* only) {
    if (check_shapes(num_q_heads, num_kv_heads, head_size, block_size)) return -2;
    int32_t group = num_q_heads / num_kv_heads;
    int bad = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        int32_t L = context_lens[s];
        double* p = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        for (int32_t h = 0; h < num_q_heads; ++h) {
            if (only && !only[(int64_t)s * num_q_heads + h]) continue;
            double* o = out + ((int64_t)s * num_q_heads + h) * head_size;
            for (int32_t d = 0; d < head_size; ++d) o[d] = 0.0;
            if (L <= 0) continue;
            int32_t kvh = h / group;
            const uint16_t* qrow = q + ((int64_t)s * num_q_heads + h) * head_size;
            double m = -INFINITY;
            for (int32_t t = 0; t < L; ++t) {
                int64_t row = pool_row(block_tables, max_blocks_per_seq, num_kv_heads, block_size,
                                       head_size, num_blocks, s, kvh, t, &bad);
                double acc = 0.0;
                if (row >= 0)
                    for (int32_t d = 0; d < head_size; ++d)
                        acc += widen(qrow[d], dtype) *
                               (or_e4m3_to_f64(k_cache[row + d]) * (double)k_scale);
                p[t] = (double)scale * acc;
                if (p[t] > m) m = p[t];
            }
            double l = 0.0;
            for (int32_t t = 0; t < L; ++t) { p[t] = exp(p[t] - m); l += p[t]; }
            for (int32_t t = 0; t < L; ++t) {
                int64_t row = pool_row(block_tables, max_blocks_per_seq, num_kv_heads, block_size,
                                       head_size, num_blocks, s, kvh, t, &bad);
                if (row < 0) continue;
                for (int32_t d = 0; d < head_size; ++d)
                    o[d] += p[t] * (or_e4m3_to_f64(v_cache[row + d]) * (double)v_scale);
            }
            for (int32_t d = 0; d < head_size; ++d) o[d] /= l;
        }
        free(p);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* Block allocator ([PR]: the v2 block manager hands out physical blocks and   */
/* the decode metadata block_tables / slot_mapping / seq_lens; [TALK]: blocks  */
/* managed like virtual-memory pages).  The written spec both sides follow:    */
/*  1. Physical ids 0..num_blocks-1 are shuffled by Fisher-Yates, for i from   */
/*     num_blocks-1 down to 1 swapping entry i with entry j = r % (i + 1),      */
/*     r the next splitmix64 output of a generator seeded with `seed`.          */
/*  2. The shuffled array is the free list; blocks are popped from its end.     */
/*  3. add_seq(id, n) pops ceil(n / block_size) blocks, in logical order.       */
/*  4. append(id) pops one block first when position len has no block yet      */
/*     (len a multiple of block_size, nothing reserved ahead), then returns the */
/*     slot of position len and increments len.                                 */
/*  5. free_seq(id) pushes the sequence's blocks back in logical order (with   */
/*     sharing: only the blocks whose reference count drops to 0).              */
/*  6. A request that needs more blocks than are free fails and changes         */
/*     nothing.                                                                */
/* ------------------------------------------------------------------------- */

/* splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014; constants of the public-domain version by S. Vigna). */
uint64_t or_splitmix64_next(uint64_t* state) {
    *state += 0x9E3779B97F4A7C15ULL;
    uint64_t z = *state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Shared prefixes ([TALK]: space sharing between requests, prefix caching).  Spec:
 *  7. Every block has a reference count: the live sequences whose table holds it.
 *     A popped block starts at 1.
 *  8. fork(src, dst, n): dst becomes live with length n <= len(src) and the first
 *     ceil(n / block_size) blocks of src, each count + 1; nothing is popped.
 *  9. Copy-on-write: when append (or reserve, see below) is about to write position
 *     len into a block whose count is > 1, it first pops a new block, records the
 *     pair (old, new) in the pending-copy list, puts the new block in the table in
 *     place of the old one and decrements the old one's count.  reserve(id, extra),
 *     extra > 0, does this to the block of position len before popping, so that a
 *     loop advanced on the device never writes into a shared block.
 * 10. take_copies returns the pending pairs in the order recorded and clears them;
 *     the caller copies those blocks on the device before writing new rows. */
typedef struct {
    int32_t num_blocks, block_size, max_seqs;
    int32_t* free_list;
    int32_t num_free;
    int32_t* refcount;     /* per physical block */
    int32_t* copies;       /* pending copy-on-write pairs (old, new) */
    int32_t ncopies, copies_cap;
    int32_t** blocks;      /* per sequence id: its physical blocks in logical order */
    int32_t* nblocks;
    int32_t* cap;
    int32_t* len;
    uint8_t* live;
} or_alloc;

or_alloc* or_alloc_create(int32_t num_blocks, int32_t block_size, uint64_t seed, int32_t max_seqs) {
    if (num_blocks <= 0 || block_size <= 0 || max_seqs <= 0) return NULL;
    or_alloc* a = (or_alloc*)calloc(1, sizeof(or_alloc));
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->max_seqs = max_seqs;
    a->free_list = (int32_t*)malloc(sizeof(int32_t) * (size_t)num_blocks);
    for (int32_t i = 0; i < num_blocks; ++i) a->free_list[i] = i;
    uint64_t st = seed;
    for (int32_t i = num_blocks - 1; i >= 1; --i) {
        uint64_t r = or_splitmix64_next(&st);
        int32_t j = (int32_t)(r % (uint64_t)(i + 1));
        int32_t tmp = a->free_list[i];
        a->free_list[i] = a->free_list[j];
        a->free_list[j] = tmp;
    }
    a->num_free = num_blocks;
    a->refcount = (int32_t*)calloc((size_t)num_blocks, sizeof(int32_t));
    a->blocks = (int32_t**)calloc((size_t)max_seqs, sizeof(int32_t*));
    a->nblocks = (int32_t*)calloc((size_t)max_seqs, sizeof(int32_t));
    a->cap = (int32_t*)calloc((size_t)max_seqs, sizeof(int32_t));
    a->len = (int32_t*)calloc((size_t)max_seqs, sizeof(int32_t));
    a->live = (uint8_t*)calloc((size_t)max_seqs, 1);
    return a;
}

void or_alloc_destroy(or_alloc* a) {
    if (!a) return;
    for (int32_t i = 0; i < a->max_seqs; ++i) free(a->blocks[i]);
    free(a->blocks); free(a->nblocks); free(a->cap); free(a->len); free(a->live);
    free(a->free_list); free(a->refcount); free(a->copies);
    free(a);
}

int32_t or_alloc_num_free(const or_alloc* a) { return a->num_free; }

static void push_block(or_alloc* a, int32_t id, int32_t phys) {
    if (a->nblocks[id] == a->cap[id]) {
        a->cap[id] = a->cap[id] ? 2 * a->cap[id] : 8;
        a->blocks[id] = (int32_t*)realloc(a->blocks[id], sizeof(int32_t) * (size_t)a->cap[id]);
    }
    a->blocks[id][a->nblocks[id]++] = phys;
}

/* Pops the next free block for sequence id (reference count 1). */
static int32_t pop_block(or_alloc* a) {
    int32_t b = a->free_list[--a->num_free];
    a->refcount[b] = 1;
    return b;
}

/* Would writing position len of id hit a shared block (rule 9)? */
static int needs_cow(const or_alloc* a, int32_t id) {
    int32_t L = a->len[id];
    int32_t logical = L / a->block_size;
    return logical < a->nblocks[id] && a->refcount[a->blocks[id][logical]] > 1;
}

static void copy_on_write(or_alloc* a, int32_t id) {
    int32_t logical = a->len[id] / a->block_size;
    int32_t old = a->blocks[id][logical];
    int32_t fresh = pop_block(a);
    a->refcount[old] -= 1;
    a->blocks[id][logical] = fresh;
    if (a->ncopies + 2 > a->copies_cap) {
        a->copies_cap = a->copies_cap ? 2 * a->copies_cap : 16;
        a->copies = (int32_t*)realloc(a->copies, sizeof(int32_t) * (size_t)a->copies_cap);
    }
    a->copies[a->ncopies++] = old;
    a->copies[a->ncopies++] = fresh;
}

/* Returns 0, -1 (bad id or already live), -3 (not enough free blocks). */
int32_t or_alloc_add_seq(or_alloc* a, int32_t id, int32_t num_tokens) {
    if (id < 0 || id >= a->max_seqs || a->live[id] || num_tokens < 0) return -1;
    int32_t need = (num_tokens + a->block_size - 1) / a->block_size;
    if (need > a->num_free) return -3;
    a->live[id] = 1;
    a->nblocks[id] = 0;
    a->len[id] = num_tokens;
    for (int32_t i = 0; i < need; ++i) push_block(a, id, pop_block(a));
    return 0;
}

/* Returns 0 and the new token's slot, -1 (unknown id), -3 (no free block). */
int32_t or_alloc_append(or_alloc* a, int32_t id, int32_t* slot) {
    if (id < 0 || id >= a->max_seqs || !a->live[id]) return -1;
    int32_t L = a->len[id];
    if (L / a->block_size >= a->nblocks[id]) {   /* position L needs a block not yet owned */
        if (a->num_free == 0) return -3;
        push_block(a, id, pop_block(a));
    } else if (needs_cow(a, id)) {               /* position L is in a shared block */
        if (a->num_free == 0) return -3;
        copy_on_write(a, id);
    }
    *slot = a->blocks[id][L / a->block_size] * a->block_size + L % a->block_size;
    a->len[id] = L + 1;
    return 0;
}

/* Lookahead reservation for a multi-step loop ([PR]: several decode steps run before the
 * scheduler sees the batch again, so their blocks must exist up front).  Spec, same on
 * both sides: reserve(id, extra) pops blocks, in logical order, until the sequence owns
 * ceil((len + extra) / block_size) blocks; len is unchanged.  Returns 0, -1, -3 (not
 * enough free blocks; nothing changed). */
int32_t or_alloc_reserve(or_alloc* a, int32_t id, int32_t extra) {
    if (id < 0 || id >= a->max_seqs || !a->live[id] || extra < 0) return -1;
    int32_t want = (a->len[id] + extra + a->block_size - 1) / a->block_size;
    int32_t need = want - a->nblocks[id];
    int32_t cow = (extra > 0 && needs_cow(a, id)) ? 1 : 0;
    if ((need > 0 ? need : 0) + cow > a->num_free) return -3;
    if (cow) copy_on_write(a, id);
    for (int32_t i = 0; i < need; ++i) push_block(a, id, pop_block(a));
    return 0;
}

/* Rule 8.  Returns 0, -1 (bad ids, dst live, src not live, n > len(src)). */
int32_t or_alloc_fork(or_alloc* a, int32_t src, int32_t dst, int32_t num_tokens) {
    if (src < 0 || src >= a->max_seqs || !a->live[src]) return -1;
    if (dst < 0 || dst >= a->max_seqs || a->live[dst] || num_tokens < 0) return -1;
    if (num_tokens > a->len[src]) return -1;
    int32_t nb = (num_tokens + a->block_size - 1) / a->block_size;
    a->live[dst] = 1;
    a->nblocks[dst] = 0;
    a->len[dst] = num_tokens;
    for (int32_t i = 0; i < nb; ++i) {
        int32_t b = a->blocks[src][i];
        a->refcount[b] += 1;
        push_block(a, dst, b);
    }
    return 0;
}

/* Rule 10.  Writes up to max_pairs (old, new) pairs; returns the number of pending
 * pairs, and takes (clears) them only if they all fit. */
int32_t or_alloc_take_copies(or_alloc* a, int32_t* pairs, int32_t max_pairs) {
    int32_t n = a->ncopies / 2;
    if (n > max_pairs) return n;
    for (int32_t i = 0; i < 2 * n; ++i) pairs[i] = a->copies[i];
    a->ncopies = 0;
    return n;
}

int32_t or_alloc_refcount(const or_alloc* a, int32_t block) {
    return (block >= 0 && block < a->num_blocks) ? a->refcount[block] : -1;
}

/* Copies whole blocks (every kv head, every row) of both pools: for each pair,
 * block `new` takes the contents of block `old`.  Bit-exact. */
int32_t or_copy_blocks(uint16_t* key_cache, uint16_t* value_cache, const int32_t* pairs,
                       int32_t n, int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                       int32_t num_blocks) {
    int64_t per = (int64_t)num_kv_heads * block_size * head_size;
    int32_t bad = 0;
    for (int32_t i = 0; i < n; ++i) {
        int32_t from = pairs[2 * i], to = pairs[2 * i + 1];
        if (from < 0 || from >= num_blocks || to < 0 || to >= num_blocks) { ++bad; continue; }
        for (int64_t e = 0; e < per; ++e) {
            key_cache[to * per + e] = key_cache[from * per + e];
            value_cache[to * per + e] = value_cache[from * per + e];
        }
    }
    return bad;
}

int32_t or_alloc_free_seq(or_alloc* a, int32_t id) {
    if (id < 0 || id >= a->max_seqs || !a->live[id]) return -1;
    for (int32_t i = 0; i < a->nblocks[id]; ++i) {
        int32_t b = a->blocks[id][i];
        if (--a->refcount[b] == 0) a->free_list[a->num_free++] = b;
    }
    a->nblocks[id] = 0;
    a->len[id] = 0;
    a->live[id] = 0;
    return 0;
}

/* Slots of positions [start, start + n) of a live sequence. */
int32_t or_alloc_slots(const or_alloc* a, int32_t id, int32_t start, int32_t n, int32_t* out) {
    if (id < 0 || id >= a->max_seqs || !a->live[id]) return -1;
    if (start < 0 || n < 0 || start + n > a->len[id]) return -1;
    for (int32_t i = 0; i < n; ++i) {
        int32_t t = start + i;
        out[i] = a->blocks[id][t / a->block_size] * a->block_size + t % a->block_size;
    }
    return 0;
}

/* Block-table rows for the listed sequences, padded with -1. */
int32_t or_alloc_block_tables(const or_alloc* a, const int32_t* ids, int32_t n,
                              int32_t max_blocks_per_seq, int32_t* out) {
    for (int32_t r = 0; r < n; ++r) {
        int32_t id = ids[r];
        if (id < 0 || id >= a->max_seqs || !a->live[id]) return -1;
        if (a->nblocks[id] > max_blocks_per_seq) return -1;
        for (int32_t c = 0; c < max_blocks_per_seq; ++c)
            out[(int64_t)r * max_blocks_per_seq + c] = c < a->nblocks[id] ? a->blocks[id][c] : -1;
    }
    return 0;
}

int32_t or_alloc_context_lens(const or_alloc* a, const int32_t* ids, int32_t n, int32_t* out) {
    for (int32_t r = 0; r < n; ++r) {
        int32_t id = ids[r];
        if (id < 0 || id >= a->max_seqs || !a->live[id]) return -1;
        out[r] = a->len[id];
    }
    return 0;
}
