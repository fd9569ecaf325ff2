/*
 * oracle.c -- plain, slow CPU reference of the paged-KV-cache attention path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file.  Only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark may load it.  It shares no code, header, table or helper with
 * the CUDA path; it has its own number-format codecs written from the format
 * definitions (IEEE 754 binary16, bfloat16 = the top half of binary32, OCP FP8
 * E4M3 "fn" variant).
 *
 * Everything is computed in double precision, one output element at a time,
 * with sums taken in the natural token order.  Results are rounded once to the
 * output format (round to nearest, ties to even).
 *
 * Sources (web pages this path is taken from):
 *  [P1] "分页注意力机制" -- translation of the vLLM PagedAttention kernel design
 *       doc (vllm.ooos.top/design/paged_attention): sections 输入参数 (inputs),
 *       概念 (concepts), Key, QK, Softmax (equation for m(x), f(x), l(x)),
 *       qk_max 和 logits (masking), Value, Output.
 *  [P2] "Paged 어텐션" (data-sketchers.com, transformers paged-attention wiki):
 *       sections "Varlen 경로" (cu_seq_lens_q/k worked example) and
 *       "Decode 경로" (block_table / cache_seqlens worked example).
 *  [P4] "Как работает paged attention? (детально)" (aivaro.ru answers/837):
 *       section 4.1 Allocation (slot of a new token), 5.1 block-wise attention.
 *  [P5] vLLM paper summary (easyvpn24.com/25506.html): section 3 解码 (decode
 *       worked example, block size 4).
 *  [P3] "ChunkLlama" (docsearch.algolia.com, vLLM feature list): "FP8 KV Cache".
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - GQA: query head h reads KV head h / (num_heads / num_kv_heads).
 *  - Masked / out-of-range tokens take no part in the max or the sum.
 *  - A query row that sees no key outputs exactly 0.
 *  - Varlen causal mask is bottom-right aligned: query i of a sequence with
 *    Lq queries and Lk keys sits at absolute position Lk - Lq + i.
 *  - FP8 KV: stored code = e4m3_satfinite_rne((float)x / scale), the division
 *    done in binary32; the stored value means code * scale.
 *  - The 1e-6 added to the softmax denominator in [P1] section exp_sum is not
 *    used: the oracle applies the exact softmax of [P1] section Softmax.
 *
 * Parity pins: every function here is checked by tests against things other
 * than itself (library codecs, torch's scaled_dot_product_attention in
 * float64, closed forms, invariants and the pages' worked examples).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* dtype codes of the oracle's own interface (numbers chosen to match the
 * public header's enum so that callers can pass the same integer; the value
 * list is an interface, not shared code) */
enum { O_F16 = 0, O_BF16 = 1, O_E4M3 = 2, O_F32 = 3 };

enum { O_OK = 0, O_ERR_ARG = 1, O_ERR_BAD_BLOCK = 6 };

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* Round x to the binary format with `p` fraction bits and minimum normal
 * exponent `emin` (gradual underflow), round-to-nearest-even.  Overflow is
 * left to the caller.  x/ulp and r*ulp are exact power-of-two scalings. */
static double round_to_format(double x, int p, int emin) {
    if (x == 0.0 || !isfinite(x)) return x;
    int E;
    frexp(fabs(x), &E); /* |x| = f * 2^E, f in [0.5, 1) */
    int e = E - 1;      /* |x| in [2^e, 2^(e+1)) */
    if (e < emin) e = emin;
    double ulp = ldexp(1.0, e - p);
    return nearbyint(x / ulp) * ulp; /* default FP environment: ties to even */
}

/* Encode an already-representable value into sign / biased exponent /
 * fraction fields. */
static uint32_t encode_fields(double r, int p, int emin, int bias, int ebits) {
    uint32_t sign = signbit(r) ? 1u : 0u;
    double a = fabs(r);
    uint32_t exp_field, frac;
    if (a == 0.0) {
        exp_field = 0;
        frac = 0;
    } else if (a < ldexp(1.0, emin)) { /* subnormal */
        exp_field = 0;
        frac = (uint32_t)(a / ldexp(1.0, emin - p));
    } else {
        int E;
        frexp(a, &E);
        int e = E - 1;
        exp_field = (uint32_t)(e + bias);
        frac = (uint32_t)((a / ldexp(1.0, e) - 1.0) * ldexp(1.0, p));
    }
    return (sign << (ebits + p)) | (exp_field << p) | frac;
}

static double decode_fields(uint32_t bits, int p, int emin, int bias, int ebits) {
    uint32_t sign = (bits >> (ebits + p)) & 1u;
    uint32_t exp_field = (bits >> p) & ((1u << ebits) - 1u);
    uint32_t frac = bits & ((1u << p) - 1u);
    double v;
    if (exp_field == 0)
        v = ldexp((double)frac, emin - p);
    else
        v = ldexp(1.0 + ldexp((double)frac, -p), (int)exp_field - bias);
    return sign ? -v : v;
}

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t h) {
    uint32_t e = (h >> 10) & 0x1f, f = h & 0x3ff;
    if (e == 0x1f) {
        if (f) return NAN;
        return (h & 0x8000) ? -INFINITY : INFINITY;
    }
    return decode_fields(h, 10, -14, 15, 5);
}

uint16_t oracle_f16_from_double(double x) {
    if (isnan(x)) return 0x7e00;
    double r = round_to_format(x, 10, -14);
    if (fabs(r) > 65504.0) return signbit(r) ? 0xfc00 : 0x7c00; /* overflow -> inf */
    return (uint16_t)encode_fields(r, 10, -14, 15, 5);
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits. */
double oracle_bf16_to_double(uint16_t b) {
    uint32_t e = (b >> 7) & 0xff, f = b & 0x7f;
    if (e == 0xff) {
        if (f) return NAN;
        return (b & 0x8000) ? -INFINITY : INFINITY;
    }
    return decode_fields(b, 7, -126, 127, 8);
}

uint16_t oracle_bf16_from_double(double x) {
    if (isnan(x)) return 0x7fc0;
    double r = round_to_format(x, 7, -126);
    double maxv = ldexp(2.0 - ldexp(1.0, -7), 127);
    if (fabs(r) > maxv) return signbit(r) ? 0xff80 : 0x7f80;
    return (uint16_t)encode_fields(r, 7, -126, 127, 8);
}

/* OCP FP8 E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 fraction bits; no
 * infinities; S.1111.111 is NaN, so the largest finite magnitude is
 * 1.75 * 2^8 = 448. */
double oracle_e4m3_to_double(uint8_t c) {
    if ((c & 0x7f) == 0x7f) return NAN;
    return decode_fields(c, 3, -6, 7, 4);
}

/* Round to nearest even, then saturate to +-448 (NaN stays NaN). */
uint8_t oracle_e4m3_from_float(float xf) {
    double x = (double)xf;
    if (isnan(x)) return 0x7f;
    double r = isinf(x) ? x : round_to_format(x, 3, -6);
    if (fabs(r) > 448.0) r = signbit(r) ? -448.0 : 448.0;
    return (uint8_t)encode_fields(r, 3, -6, 7, 4);
}

static double load_elem(const void* base, int dtype, int64_t i) {
    switch (dtype) {
    case O_F16: return oracle_f16_to_double(((const uint16_t*)base)[i]);
    case O_BF16: return oracle_bf16_to_double(((const uint16_t*)base)[i]);
    case O_E4M3: return oracle_e4m3_to_double(((const uint8_t*)base)[i]);
    case O_F32: return (double)((const float*)base)[i];
    default: return NAN;
    }
}

static void store_elem(void* base, int dtype, int64_t i, double v) {
    switch (dtype) {
    case O_F16: ((uint16_t*)base)[i] = oracle_f16_from_double(v); break;
    case O_BF16: ((uint16_t*)base)[i] = oracle_bf16_from_double(v); break;
    case O_F32: ((float*)base)[i] = (float)v; break;
    default: break;
    }
}

static int elem_bytes(int dtype) {
    return dtype == O_E4M3 ? 1 : (dtype == O_F32 ? 4 : 2);
}

/* ------------------------------------------------------------------------ */
/* Slot of a new token ([P4] section 4.1; [P5] section 3)                    */
/* ------------------------------------------------------------------------ */

/* For token i of sequence seq_idx[i] at position pos[i]: the logical block is
 * pos / block_size, the physical block is block_table[seq][logical], and the
 * slot is physical * block_size + pos % block_size.  An unmapped entry (< 0)
 * yields slot -1. */
void oracle_slot_mapping(const int32_t* block_table, int32_t max_blocks, int32_t block_size,
                         const int32_t* seq_idx, const int64_t* pos, int64_t n,
                         int64_t* slots_out) {
    for (int64_t i = 0; i < n; ++i) {
        int64_t logical = pos[i] / block_size;
        int64_t offset = pos[i] % block_size;
        int32_t phys = logical < max_blocks ? block_table[(int64_t)seq_idx[i] * max_blocks + logical] : -1;
        slots_out[i] = phys < 0 ? -1 : (int64_t)phys * block_size + offset;
    }
}

/* ------------------------------------------------------------------------ */
/* Cache layout: [num_blocks][num_kv_heads][block_size][head_size]          */
/* ------------------------------------------------------------------------ */

static int64_t cache_index(int64_t blk, int64_t h, int64_t off, int64_t d,
                           int64_t num_kv_heads, int64_t block_size, int64_t head_size) {
    return ((blk * num_kv_heads + h) * block_size + off) * head_size + d;
}

/* Write of new K/V rows into their slots ([P2] Decode 경로: the cache is
 * updated in place through the block table; [P4] 4.1 step 5; [P5] 3).
 * k, v: [T][num_kv_heads][head_size] with `token_stride` elements between
 * tokens.  slot < 0 skips the token.  Same-dtype writes move bits unchanged;
 * an E4M3 cache stores e4m3_satfinite_rne((float)x / scale). */
int oracle_cache_write(void* k_cache, void* v_cache, int kv_dtype, int64_t num_blocks,
                       int32_t block_size, int32_t num_kv_heads, int32_t head_size,
                       float k_scale, float v_scale, const void* k, const void* v,
                       int in_dtype, int64_t num_tokens, int64_t token_stride,
                       const int64_t* slot_mapping) {
    if (kv_dtype != O_E4M3 && kv_dtype != in_dtype) return O_ERR_ARG;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        int64_t blk = slot / block_size, off = slot % block_size;
        if (blk >= num_blocks) return O_ERR_BAD_BLOCK;
        for (int64_t h = 0; h < num_kv_heads; ++h) {
            for (int64_t d = 0; d < head_size; ++d) {
                int64_t src = t * token_stride + h * head_size + d;
                int64_t dst = cache_index(blk, h, off, d, num_kv_heads, block_size, head_size);
                if (kv_dtype == O_E4M3) {
                    float xk = (float)load_elem(k, in_dtype, src);
                    float xv = (float)load_elem(v, in_dtype, src);
                    volatile float qk = xk / k_scale; /* binary32 IEEE division */
                    volatile float qv = xv / v_scale;
                    ((uint8_t*)k_cache)[dst] = oracle_e4m3_from_float(qk);
                    ((uint8_t*)v_cache)[dst] = oracle_e4m3_from_float(qv);
                } else {
                    ((uint16_t*)k_cache)[dst] = ((const uint16_t*)k)[src];
                    ((uint16_t*)v_cache)[dst] = ((const uint16_t*)v)[src];
                }
            }
        }
    }
    return O_OK;
}

/* Copy whole physical blocks (copy-on-write of a shared block, [P4] 3.3). */
int oracle_copy_blocks(void* k_cache, void* v_cache, int kv_dtype, int64_t num_blocks,
                       int32_t block_size, int32_t num_kv_heads, int32_t head_size,
                       const int32_t* pairs, int32_t n) {
    int64_t bytes = (int64_t)num_kv_heads * block_size * head_size * elem_bytes(kv_dtype);
    for (int32_t i = 0; i < n; ++i) {
        int64_t s = pairs[2 * i], d = pairs[2 * i + 1];
        if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) return O_ERR_BAD_BLOCK;
        memmove((char*)k_cache + d * bytes, (char*)k_cache + s * bytes, (size_t)bytes);
        memmove((char*)v_cache + d * bytes, (char*)v_cache + s * bytes, (size_t)bytes);
    }
    return O_OK;
}

/* ------------------------------------------------------------------------ */
/* Attention of one query row over the first `nkeys` logical keys of one     */
/* sequence, gathered page by page through its block-table row.             */
/* ------------------------------------------------------------------------ */

typedef struct {
    const void *k_cache, *v_cache;
    int kv_dtype;
    double k_scale, v_scale;
    int64_t num_blocks;
    int32_t block_size, num_kv_heads, head_size;
} cache_view;

/* scores s_t = scale * sum_d q_d K[t][d]  ([P1] QK);
 * softmax by max subtraction: m = max s, f_t = exp(s_t - m), l = sum f,
 * p = f / l  ([P1] Softmax equation);  o_d = sum_t p_t V[t][d]  ([P1] Value).
 * Keys are reached as K_b[t] = cache[block_table[t / bs]][kvh][t % bs][:]
 * ([P1] Key; [P2] Decode 경로).  Returns O_ERR_BAD_BLOCK for a table entry
 * outside [0, num_blocks) among the entries the keys need. */
static int attend_row(const cache_view* c, const int32_t* table_row, int32_t kvh,
                      const double* q, int64_t nkeys, double scale, double* o, double* s) {
    int64_t D = c->head_size, bs = c->block_size;
    for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
    if (nkeys <= 0) return O_OK; /* no visible key: output 0 */
    for (int64_t t = 0; t < nkeys; ++t) {
        int32_t blk = table_row[t / bs];
        if (blk < 0 || blk >= c->num_blocks) return O_ERR_BAD_BLOCK;
    }
    double m = -INFINITY;
    for (int64_t t = 0; t < nkeys; ++t) {
        int64_t blk = table_row[t / bs], off = t % bs;
        double acc = 0.0;
        for (int64_t d = 0; d < D; ++d) {
            double kd = load_elem(c->k_cache, c->kv_dtype,
                                  cache_index(blk, kvh, off, d, c->num_kv_heads, bs, D));
            if (c->kv_dtype == O_E4M3) kd *= c->k_scale;
            acc += q[d] * kd;
        }
        s[t] = scale * acc;
        if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (int64_t t = 0; t < nkeys; ++t) {
        s[t] = exp(s[t] - m);
        l += s[t];
    }
    for (int64_t t = 0; t < nkeys; ++t) {
        int64_t blk = table_row[t / bs], off = t % bs;
        double p = s[t] / l;
        for (int64_t d = 0; d < D; ++d) {
            double vd = load_elem(c->v_cache, c->kv_dtype,
                                  cache_index(blk, kvh, off, d, c->num_kv_heads, bs, D));
            if (c->kv_dtype == O_E4M3) vd *= c->v_scale;
            o[d] += p * vd;
        }
    }
    return O_OK;
}

static int set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

int oracle_num_threads(int nthreads) { return set_threads(nthreads); }

/* Single-query decode ([P1] whole kernel walk-through; [P2] Decode 경로).
 * q:   [num_seqs][num_heads][head_size] in q_dtype
 * out: [num_seqs][num_heads][head_size] in q_dtype (rounded once), and, when
 *      out_f64 is not NULL, the unrounded double result as well.
 * seq_lens[b] is the attended length L_b; keys t < L_b take part.
 * Returns O_ERR_ARG if num_heads % num_kv_heads != 0, O_ERR_BAD_BLOCK for a bad
 * block id among the entries a sequence needs. */
int oracle_decode(void* out, double* out_f64, const void* q, int q_dtype,
                  const void* k_cache, const void* v_cache, int kv_dtype,
                  double k_scale, double v_scale, int64_t num_blocks, int32_t block_size,
                  int32_t num_kv_heads, int32_t head_size, const int32_t* block_table,
                  int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                  int32_t num_heads, double scale, int nthreads) {
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return O_ERR_ARG;
    for (int32_t b = 0; b < num_seqs; ++b)
        if (seq_lens[b] < 0 || (int64_t)seq_lens[b] > (int64_t)max_blocks_per_seq * block_size)
            return O_ERR_ARG;
    set_threads(nthreads);
    cache_view c = {k_cache, v_cache, kv_dtype, k_scale, v_scale, num_blocks,
                    block_size, num_kv_heads, head_size};
    int32_t group = num_heads / num_kv_heads;
    int64_t D = head_size;
    int status = O_OK;
    int64_t total = (int64_t)num_seqs * num_heads;
#pragma omp parallel
    {
        int64_t maxlen = 1;
        for (int32_t b = 0; b < num_seqs; ++b)
            if (seq_lens[b] > maxlen) maxlen = seq_lens[b];
        double* qd = (double*)malloc(sizeof(double) * D);
        double* o = (double*)malloc(sizeof(double) * D);
        double* s = (double*)malloc(sizeof(double) * maxlen);
#pragma omp for schedule(dynamic, 1)
        for (int64_t bh = 0; bh < total; ++bh) {
            int64_t b = bh / num_heads, h = bh % num_heads;
            for (int64_t d = 0; d < D; ++d) qd[d] = load_elem(q, q_dtype, bh * D + d);
            int rc = attend_row(&c, block_table + b * max_blocks_per_seq, (int32_t)(h / group),
                                qd, seq_lens[b], scale, o, s);
            if (rc != O_OK) {
#pragma omp critical
                status = rc;
            }
            for (int64_t d = 0; d < D; ++d) {
                if (out) store_elem(out, q_dtype, bh * D + d, o[d]);
                if (out_f64) out_f64[bh * D + d] = o[d];
            }
        }
        free(qd);
        free(o);
        free(s);
    }
    return status;
}

/* Varlen prefill over the paged cache ([P2] Varlen 경로: cu_seq_lens_q/k index
 * the packed queries and give each sequence's key count; keys are read from
 * the paged cache through block_table as in [P2] Decode 경로; [P4] 5.1: causal
 * masking per block).
 * q, out: [total_q][num_heads][head_size], sequence b owns rows
 *         cu_seq_lens_q[b] .. cu_seq_lens_q[b+1]-1.
 * Lk_b = cu_seq_lens_k[b+1] - cu_seq_lens_k[b] keys at logical positions 0..Lk_b-1.
 * causal: query i sees key j iff j <= i + Lk_b - Lq_b (bottom-right aligned). */
int oracle_prefill(void* out, double* out_f64, const void* q, int q_dtype,
                   const void* k_cache, const void* v_cache, int kv_dtype, double k_scale,
                   double v_scale, int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                   int32_t head_size, const int32_t* block_table, int32_t max_blocks_per_seq,
                   const int32_t* cu_seq_lens_q, const int32_t* cu_seq_lens_k, int32_t num_seqs,
                   int32_t num_heads, double scale, int causal, int nthreads) {
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return O_ERR_ARG;
    for (int32_t b = 0; b < num_seqs; ++b) {
        int64_t lq = cu_seq_lens_q[b + 1] - cu_seq_lens_q[b];
        int64_t lk = cu_seq_lens_k[b + 1] - cu_seq_lens_k[b];
        if (lq < 0 || lk < 0 || lk > (int64_t)max_blocks_per_seq * block_size) return O_ERR_ARG;
    }
    set_threads(nthreads);
    cache_view c = {k_cache, v_cache, kv_dtype, k_scale, v_scale, num_blocks,
                    block_size, num_kv_heads, head_size};
    int32_t group = num_heads / num_kv_heads;
    int64_t D = head_size;
    int64_t total_q = cu_seq_lens_q[num_seqs];
    int status = O_OK;
    int64_t rows = total_q * num_heads;
#pragma omp parallel
    {
        int64_t maxlen = 1;
        for (int32_t b = 0; b < num_seqs; ++b) {
            int64_t lk = cu_seq_lens_k[b + 1] - cu_seq_lens_k[b];
            if (lk > maxlen) maxlen = lk;
        }
        double* qd = (double*)malloc(sizeof(double) * D);
        double* o = (double*)malloc(sizeof(double) * D);
        double* s = (double*)malloc(sizeof(double) * maxlen);
#pragma omp for schedule(dynamic, 4)
        for (int64_t rh = 0; rh < rows; ++rh) {
            int64_t row = rh / num_heads, h = rh % num_heads;
            int32_t b = 0; /* the sequence whose query rows contain `row` */
            while (cu_seq_lens_q[b + 1] <= row) ++b;
            int64_t lq = cu_seq_lens_q[b + 1] - cu_seq_lens_q[b];
            int64_t lk = cu_seq_lens_k[b + 1] - cu_seq_lens_k[b];
            int64_t i = row - cu_seq_lens_q[b];
            int64_t nkeys = lk;
            if (causal) {
                int64_t last = i + lk - lq; /* last visible key position */
                nkeys = last + 1 < lk ? last + 1 : lk;
            }
            for (int64_t d = 0; d < D; ++d) qd[d] = load_elem(q, q_dtype, rh * D + d);
            int rc = attend_row(&c, block_table + (int64_t)b * max_blocks_per_seq,
                                (int32_t)(h / group), qd, nkeys, scale, o, s);
            if (rc != O_OK) {
#pragma omp critical
                status = rc;
            }
            for (int64_t d = 0; d < D; ++d) {
                if (out) store_elem(out, q_dtype, rh * D + d, o[d]);
                if (out_f64) out_f64[rh * D + d] = o[d];
            }
        }
        free(qd);
        free(o);
        free(s);
    }
    return status;
}

/* Brute-force attention over explicit dense rows (no paging), double in and
 * out.  q: [lq][D], k, v: [lk][D].  With `causal` set, query i sees keys
 * j <= i + causal_shift (the shift may be negative); otherwise all keys.
 * Used only to test the paged functions above. */
void oracle_attention_dense(double* out, const double* q, const double* k, const double* v,
                            int64_t lq, int64_t lk, int64_t D, double scale, int causal,
                            int64_t causal_shift) {
    double* s = (double*)malloc(sizeof(double) * (lk > 0 ? lk : 1));
    for (int64_t i = 0; i < lq; ++i) {
        int64_t n = lk;
        if (causal && i + causal_shift + 1 < n) n = i + causal_shift + 1;
        for (int64_t d = 0; d < D; ++d) out[i * D + d] = 0.0;
        if (n <= 0) continue;
        double m = -INFINITY;
        for (int64_t j = 0; j < n; ++j) {
            double a = 0.0;
            for (int64_t d = 0; d < D; ++d) a += q[i * D + d] * k[j * D + d];
            s[j] = scale * a;
            if (s[j] > m) m = s[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            s[j] = exp(s[j] - m);
            l += s[j];
        }
        for (int64_t j = 0; j < n; ++j)
            for (int64_t d = 0; d < D; ++d) out[i * D + d] += s[j] / l * v[j * D + d];
    }
    free(s);
}
