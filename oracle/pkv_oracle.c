/*
 * pkv_oracle.c — FP64 CPU oracle for one paged-KV decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or helper with the CUDA
 * path: it reads the documented pool layout with its own loops.
 *
 * What it computes, and where each step comes from:
 *
 *   - The KV page pool and block table: tinyllm, "The repository currently
 *     provides" (a runner-owned physical KV page pool with a logical block
 *     table per active sequence) and "Known limitations" (16-token pages).
 *   - KV storage as f16, bf16, f32 and q8/q8_0: Leone, "What ships" (f32, f16 and q8 KV
 *     storage); tinyllm, "The repository currently provides" (BF16/F32 KV
 *     caching); LeatEngine, "Run" (--cache-type q8_0 keeps the KV cache the
 *     way llama.cpp's q8_0 cache does, in about half the memory of f16).
 *     q8_0 here: blocks of 32 consecutive head_dim values, one f16 scale per
 *     block, d = amax/127, codes round(x/d) with ties away from zero.
 *   - Decode attention with GQA: tinyllm, "The repository currently provides"
 *     (28-layer model with GQA attention; causal attention with contiguous and
 *     paged-reference cache paths).  One query token per row attends to all
 *     of that row's cached tokens: out = softmax(scale * q K^T) V.
 *   - The gather strategy: tinyllm, "Known limitations" (the paged-reference
 *     decode gathers a row's logical pages and then runs dense attention).
 *     The oracle does the same: it walks the block table token by token and
 *     evaluates the dense formula in double precision.
 *   - Variable-length batched decode: tinyllm, "The repository currently
 *     provides" (variable-length batched decode for several active
 *     sequences); Leone, "What ships" (continuous decode batching).
 *   - Sliding-window KV caches: LeatEngine, "Capabilities".  Reading: with a
 *     window W > 0 a row of L tokens attends to its last W tokens,
 *     [max(0, L - W), L), the new token included; W = 0 means all L.
 *   - Several query tokens per row (Leone, "What ships": chunked prefill and
 *     exact speculative verification; LeatEngine, "Capabilities": chunked
 *     prefill, speculative decoding).  Reading: a row of L tokens whose last
 *     q_len are new has one query per new token; query j sits at position
 *     P = L - q_len + j and attends causally to [a, P + 1), a = max(0,
 *     P + 1 - W) under a window W (0 otherwise).
 *
 * Readings where the pages are silent (each is restated where it is used):
 *   - GQA head map: query head g reads KV head g / (n_q_heads / n_kv_heads).
 *   - seq_lens counts the attended tokens including the one appended this
 *     step; the append writes position seq_lens[i] - 1.
 *   - Pool layout per layer: data [page][kv_head][slot 0..15][head_dim];
 *     q8_0 scales [page][kv_head][slot][head_dim / 32] (f16 bits).
 *   - q8_0 rounding: d = fl32(amax / 127) by IEEE division; the stored scale
 *     is f16(d) rounded to nearest even; each code is round_half_away(fl32(x /
 *     d)) computed with the fp32 d; amax == 0 gives d = 0 and all codes 0.
 *
 * fp32 division emulated in double: (float)((double)a / (double)b) equals the
 * correctly rounded fp32 quotient, because rounding a quotient first to 53 bits
 * and then to 24 bits is innocuous when 53 >= 2*24 + 2 (S. A. Figueroa, "When
 * is double rounding innocuous?", SIGNUM Newsletter 30(3), 1995).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef M_LOG2E
#define M_LOG2E 1.4426950408889634074
#endif

#define ORACLE_PAGE 16 /* tokens per physical page (tinyllm, Known limitations) */
#define ORACLE_QBLOCK 32 /* q8_0 block length along head_dim */

enum { ORACLE_F16 = 0, ORACLE_Q8_0 = 1, ORACLE_BF16 = 2, ORACLE_F32 = 3 };
enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_BAD_PAGE = 2 };

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the following parallel loops (timing only: results do not
 * depend on it, every output element is computed by one thread). */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------ f16 --- */

/* Exact value of an IEEE binary16 bit pattern, widened to double.
 * Fields: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24); /* subnormal: frac * 2^-24 */
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), expo - 25); /* (1.frac) * 2^(expo-15) */
    return sign ? -mag : mag;
}

/* Round an fp32 value to the nearest binary16, ties to even (IEEE 754
 * roundTiesToEven), returning its bit pattern.  Written from the definition:
 * find the spacing (ulp) of binary16 numbers at |x|, count whole ulps, and
 * round the remainder.  Values whose rounded magnitude reaches 65520 overflow
 * to infinity (65504 is the largest finite binary16; 65520 is the midpoint to
 * the next power of two and ties to the even side, which is infinity). */
uint16_t oracle_f16_from_f32(float xf) {
    double x = (double)xf; /* exact */
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7e00);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
    double ulp;
    if (a < ldexp(1.0, -14)) {
        ulp = ldexp(1.0, -24); /* subnormal range: fixed spacing 2^-24 */
    } else {
        int e;
        frexp(a, &e);          /* a = m * 2^e with m in [0.5, 1) */
        ulp = ldexp(1.0, e - 11); /* 11 significant bits in [2^(e-1), 2^e) */
    }
    double n = a / ulp;      /* exact: power-of-two scaling */
    double whole = floor(n);
    double rem = n - whole;  /* exact */
    if (rem > 0.5 || (rem == 0.5 && fmod(whole, 2.0) != 0.0)) whole += 1.0;
    double r = whole * ulp;  /* the rounded magnitude, <= 65504 here */
    if (r == 0.0) return sign;
    if (r < ldexp(1.0, -14))
        return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -24)));
    int e;
    double m = frexp(r, &e); /* r = m * 2^e, m in [0.5, 1) */
    int expo = e - 1 + 15;
    int frac = (int)((2.0 * m - 1.0) * 1024.0);
    return (uint16_t)(sign | (expo << 10) | frac);
}

/* ----------------------------------------------------------------- bf16 --- */

/* Exact value of a bfloat16 bit pattern (the high half of a binary32: 1 sign
 * bit, 8 exponent bits with bias 127, 7 fraction bits), widened to double. */
double oracle_bf16_to_f64(uint16_t b) {
    int sign = (b >> 15) & 1;
    int expo = (b >> 7) & 0xff;
    int frac = b & 0x7f;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -133); /* subnormal: frac * 2^(1-127-7) */
    else if (expo == 255)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(128 + frac), expo - 134); /* (1.frac) * 2^(expo-127) */
    return sign ? -mag : mag;
}

/* Round an fp32 value to the nearest bfloat16, ties to even, returning its
 * bit pattern; written from the definition like the binary16 rounding above:
 * 8 significant bits, spacing 2^-133 below 2^-126, and magnitudes that round
 * to 2^128 (the midpoint (2 - 2^-8) * 2^127 included: it ties to the even
 * side, the infinity) overflow to infinity. */
uint16_t oracle_bf16_from_f32(float xf) {
    double x = (double)xf; /* exact */
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7fc0);
    if (a >= ldexp(2.0 - ldexp(1.0, -8), 127)) return (uint16_t)(sign | 0x7f80);
    double ulp;
    if (a < ldexp(1.0, -126)) {
        ulp = ldexp(1.0, -133);
    } else {
        int e;
        frexp(a, &e);            /* a in [2^(e-1), 2^e) */
        ulp = ldexp(1.0, e - 8); /* 8 significant bits */
    }
    double n = a / ulp;
    double whole = floor(n);
    double rem = n - whole;
    if (rem > 0.5 || (rem == 0.5 && fmod(whole, 2.0) != 0.0)) whole += 1.0;
    double r = whole * ulp;
    if (r == 0.0) return sign;
    if (r < ldexp(1.0, -126)) return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -133)));
    int e;
    double m = frexp(r, &e);     /* r = m * 2^e, m in [0.5, 1) */
    int expo = e - 1 + 127;
    int frac = (int)((2.0 * m - 1.0) * 128.0);
    return (uint16_t)(sign | (expo << 7) | frac);
}

/* Encode n fp32 values to bfloat16 bit patterns. */
void oracle_bf16_encode(const float *x, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_from_f32(x[i]);
}

/* ----------------------------------------------------------------- q8_0 --- */

/* Round half away from zero, on a value whose magnitude is far below 2^52. */
static double round_half_away(double y) {
    return y < 0.0 ? -floor(-y + 0.5) : floor(y + 0.5);
}

/* Correctly rounded fp32 quotient a / b (see the double-rounding note above). */
static float fdiv32(float a, float b) { return (float)((double)a / (double)b); }

/* Encode one block of 32 fp32 values as q8_0: the f16 scale bits and 32
 * int8 codes.  Returns the fp32 scale d used for the codes. */
float oracle_q8_0_encode_block(const float *x, int8_t *codes, uint16_t *scale_bits) {
    float amax = 0.0f;
    for (int i = 0; i < ORACLE_QBLOCK; ++i) {
        float ax = fabsf(x[i]);
        if (ax > amax) amax = ax;
    }
    float d = fdiv32(amax, 127.0f);
    *scale_bits = oracle_f16_from_f32(d);
    for (int i = 0; i < ORACLE_QBLOCK; ++i) {
        double c = 0.0;
        if (d != 0.0f) c = round_half_away((double)fdiv32(x[i], d));
        if (c > 127.0) c = 127.0;   /* cannot trigger: |x| <= amax */
        if (c < -127.0) c = -127.0;
        codes[i] = (int8_t)c;
    }
    return d;
}

/* Encode a whole array of n fp32 values (n a multiple of 32) block by block:
 * codes[n], scale_bits[n / 32]. Used to fill a pool from fp32 context values. */
void oracle_q8_0_encode(const float *x, int64_t n, int8_t *codes, uint16_t *scale_bits) {
    for (int64_t b = 0; b < n / ORACLE_QBLOCK; ++b)
        oracle_q8_0_encode_block(x + b * ORACLE_QBLOCK, codes + b * ORACLE_QBLOCK,
                                 scale_bits + b);
}

/* Encode n fp32 values to f16 bit patterns. */
void oracle_f16_encode(const float *x, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_from_f32(x[i]);
}

/* ------------------------------------------------------------ the pool --- */

/* Stored value of element d of slot `slot` of (page, kv_head), widened to
 * double.  f16 / bf16: the binary16 / bfloat16 value.  f32: the binary32
 * value (stored as given, no rounding).  q8_0: f16 scale of the element's
 * block times its int8 code.  Layout per layer (a reading; the pages fix
 * none):
 *   data   [num_pages][n_kv][16][D]        (f16 or bf16 bits, binary32, or int8 codes)
 *   scales [num_pages][n_kv][16][D / 32]   (f16 bits; q8_0 only)           */
static double stored(int dtype, const void *data, const uint16_t *scales, int n_kv,
                     int D, int64_t page, int kvh, int slot, int d) {
    int64_t row = (page * n_kv + kvh) * ORACLE_PAGE + slot;
    if (dtype == ORACLE_F16) return oracle_f16_to_f64(((const uint16_t *)data)[row * D + d]);
    if (dtype == ORACLE_BF16) return oracle_bf16_to_f64(((const uint16_t *)data)[row * D + d]);
    if (dtype == ORACLE_F32) return (double)((const float *)data)[row * D + d];
    double sc = oracle_f16_to_f64(scales[row * (D / ORACLE_QBLOCK) + d / ORACLE_QBLOCK]);
    return sc * (double)((const int8_t *)data)[row * D + d];
}

/* Physical page holding logical token t of row i, through the block table;
 * -1 if the table entry is outside the pool. */
static int64_t page_of(const int32_t *block_table, int bt_stride, int i, int t, int num_pages) {
    int32_t p = block_table[(int64_t)i * bt_stride + t / ORACLE_PAGE];
    return (p >= 0 && p < num_pages) ? p : -1;
}

/* Store one fp32 K and V vector (D values each) of KV head h at position pos
 * of row i. */
static int store_token(int dtype, int n_kv, int D, const float *kx, const float *vx,
                       const int32_t *block_table, int bt_stride, int i, int h, int pos,
                       int num_pages, void *k_data, void *v_data, uint16_t *k_scales,
                       uint16_t *v_scales) {
    if (pos / ORACLE_PAGE >= bt_stride) return ORACLE_BAD_PAGE;
    int64_t page = page_of(block_table, bt_stride, i, pos, num_pages);
    if (page < 0) return ORACLE_BAD_PAGE;
    int64_t row = (page * n_kv + h) * ORACLE_PAGE + pos % ORACLE_PAGE;
    if (dtype == ORACLE_F16) {
        oracle_f16_encode(kx, D, (uint16_t *)k_data + row * D);
        oracle_f16_encode(vx, D, (uint16_t *)v_data + row * D);
    } else if (dtype == ORACLE_BF16) {
        oracle_bf16_encode(kx, D, (uint16_t *)k_data + row * D);
        oracle_bf16_encode(vx, D, (uint16_t *)v_data + row * D);
    } else if (dtype == ORACLE_F32) {  /* stored as given */
        memcpy((float *)k_data + row * D, kx, (size_t)D * sizeof(float));
        memcpy((float *)v_data + row * D, vx, (size_t)D * sizeof(float));
    } else {
        oracle_q8_0_encode(kx, D, (int8_t *)k_data + row * D, k_scales + row * (D / ORACLE_QBLOCK));
        oracle_q8_0_encode(vx, D, (int8_t *)v_data + row * D, v_scales + row * (D / ORACLE_QBLOCK));
    }
    return ORACLE_OK;
}

/* Several new tokens per row: k_new, v_new fp32 [rows][q_len][n_kv][D];
 * token j of row i (L = seq_lens[i] >= q_len, the length after the step)
 * goes to position L - q_len + j.  Rows with L <= 0 write nothing. */
int oracle_kv_append_mq(int dtype, int num_rows, int q_len, int n_kv, int D, const float *k_new,
                        const float *v_new, const int32_t *block_table, int bt_stride,
                        const int32_t *seq_lens, int num_pages, void *k_data, void *v_data,
                        uint16_t *k_scales, uint16_t *v_scales) {
    if (D % ORACLE_QBLOCK || q_len < 1) return ORACLE_BAD_ARG;
    for (int i = 0; i < num_rows; ++i) {
        int L = seq_lens[i];
        if (L <= 0) continue;
        if (L < q_len) return ORACLE_BAD_ARG;
        for (int j = 0; j < q_len; ++j)
            for (int h = 0; h < n_kv; ++h) {
                int64_t src = (((int64_t)i * q_len + j) * n_kv + h) * D;
                int st = store_token(dtype, n_kv, D, k_new + src, v_new + src, block_table,
                                     bt_stride, i, h, L - q_len + j, num_pages, k_data, v_data,
                                     k_scales, v_scales);
                if (st != ORACLE_OK) return st;
            }
    }
    return ORACLE_OK;
}

/* kv_append: write each row's new K and V token (fp32 [rows][n_kv][D]) into
 * page block_table[i][(L-1)/16], slot (L-1)%16, with L = seq_lens[i] (the
 * length after this token).  Rows with L <= 0 write nothing. */
int oracle_kv_append(int dtype, int num_rows, int n_kv, int D, const float *k_new,
                     const float *v_new, const int32_t *block_table, int bt_stride,
                     const int32_t *seq_lens, int num_pages, void *k_data, void *v_data,
                     uint16_t *k_scales, uint16_t *v_scales) {
    if (D % ORACLE_QBLOCK) return ORACLE_BAD_ARG;
    for (int i = 0; i < num_rows; ++i) {
        int L = seq_lens[i];
        if (L <= 0) continue;
        int pos = L - 1;
        if (pos / ORACLE_PAGE >= bt_stride) return ORACLE_BAD_PAGE;
        int64_t page = page_of(block_table, bt_stride, i, pos, num_pages);
        if (page < 0) return ORACLE_BAD_PAGE;
        int slot = pos % ORACLE_PAGE;
        for (int h = 0; h < n_kv; ++h) {
            int64_t row = (page * n_kv + h) * ORACLE_PAGE + slot;
            const float *kx = k_new + ((int64_t)i * n_kv + h) * D;
            const float *vx = v_new + ((int64_t)i * n_kv + h) * D;
            if (dtype == ORACLE_F16) {
                oracle_f16_encode(kx, D, (uint16_t *)k_data + row * D);
                oracle_f16_encode(vx, D, (uint16_t *)v_data + row * D);
            } else if (dtype == ORACLE_BF16) {
                oracle_bf16_encode(kx, D, (uint16_t *)k_data + row * D);
                oracle_bf16_encode(vx, D, (uint16_t *)v_data + row * D);
            } else if (dtype == ORACLE_F32) {  /* the fp32 values, unrounded */
                memcpy((float *)k_data + row * D, kx, (size_t)D * sizeof(float));
                memcpy((float *)v_data + row * D, vx, (size_t)D * sizeof(float));
            } else {
                oracle_q8_0_encode(kx, D, (int8_t *)k_data + row * D,
                                   k_scales + row * (D / ORACLE_QBLOCK));
                oracle_q8_0_encode(vx, D, (int8_t *)v_data + row * D,
                                   v_scales + row * (D / ORACLE_QBLOCK));
            }
        }
    }
    return ORACLE_OK;
}

/* Scores s_t = scale * <q, K_t> for tokens t in [t0, t1) of row i, KV head h.
 * Returns 0, or ORACLE_BAD_PAGE if the table points outside the pool. */
static int scores(int dtype, const void *k_data, const uint16_t *k_scales, int n_kv, int D,
                  const int32_t *block_table, int bt_stride, int num_pages, int i, int h,
                  const float *q, double scale, int t0, int t1, double *s) {
    for (int t = t0; t < t1; ++t) {
        int64_t page = page_of(block_table, bt_stride, i, t, num_pages);
        if (page < 0) return ORACLE_BAD_PAGE;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += (double)q[d] * stored(dtype, k_data, k_scales, n_kv, D, page, h,
                                         t % ORACLE_PAGE, d);
        s[t - t0] = scale * dot;
    }
    return ORACLE_OK;
}

/* First attended token of a row of L tokens under a window W (0: none). */
static int window_start(int L, int window) { return window > 0 && L > window ? L - window : 0; }

/* Attention of one query vector q (D values) of row i over KV head h's
 * tokens [a, b), b > a: o = sum_t softmax_t(scale <q, K_t>) V_t, in double
 * with the maximum subtracted before exp. */
static int attend(int dtype, const void *k_data, const void *v_data, const uint16_t *k_scales,
                  const uint16_t *v_scales, int n_kv, int D, const int32_t *block_table,
                  int bt_stride, int num_pages, int i, int h, const float *q, double scale,
                  int a, int b, double *o) {
    const int n = b - a;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    if (!s) return ORACLE_BAD_ARG;
    if (scores(dtype, k_data, k_scales, n_kv, D, block_table, bt_stride, num_pages, i, h, q,
               scale, a, b, s) != ORACLE_OK) {
        free(s);
        return ORACLE_BAD_PAGE;
    }
    double m = -INFINITY;
    for (int t = 0; t < n; ++t) m = s[t] > m ? s[t] : m;
    double l = 0.0;
    for (int t = a; t < b; ++t) {
        double p = exp(s[t - a] - m);
        l += p;
        int64_t page = page_of(block_table, bt_stride, i, t, num_pages);
        for (int d = 0; d < D; ++d)
            o[d] += p * stored(dtype, v_data, v_scales, n_kv, D, page, h, t % ORACLE_PAGE, d);
    }
    for (int d = 0; d < D; ++d) o[d] /= l;
    free(s);
    return ORACLE_OK;
}

/* Decode attention for every row and query head:
 *   out[i][g] = sum_{a_i <= t < L_i} softmax_t(scale * <q[i][g], K[i][h][t]>) V[i][h][t]
 * with h = g / (n_q / n_kv), a_i = max(0, L_i - window) (a_i = 0 for window
 * 0), K and V the stored values gathered through the block table, evaluated
 * in double with the maximum subtracted before exp.  Rows with L_i <= 0
 * produce zeros.  out is double [rows][n_q][D]. */
int oracle_decode_attention(int dtype, int num_rows, int n_q, int n_kv, int D, const float *q,
                            const void *k_data, const void *v_data, const uint16_t *k_scales,
                            const uint16_t *v_scales, const int32_t *block_table,
                            int bt_stride, const int32_t *seq_lens, int num_pages,
                            double scale, int window, double *out) {
    if (n_kv <= 0 || n_q % n_kv || D % ORACLE_QBLOCK || window < 0) return ORACLE_BAD_ARG;
    for (int i = 0; i < num_rows; ++i)
        if (seq_lens[i] > (int64_t)bt_stride * ORACLE_PAGE) return ORACLE_BAD_ARG;
    const int group = n_q / n_kv;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t ig = 0; ig < (int64_t)num_rows * n_q; ++ig) {
        int i = (int)(ig / n_q), g = (int)(ig % n_q), h = g / group;
        int L = seq_lens[i];
        double *o = out + ig * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (L <= 0) continue;
        if (attend(dtype, k_data, v_data, k_scales, v_scales, n_kv, D, block_table, bt_stride,
                   num_pages, i, h, q + ig * D, scale, window_start(L, window), L, o) != ORACLE_OK) {
#pragma omp atomic write
            status = ORACLE_BAD_PAGE;
        }
    }
    return status;
}

/* Several queries per row: q and out are [rows][q_len][n_q][D]; query j of
 * row i (L = seq_lens[i] >= q_len) sits at position P = L - q_len + j and
 * attends to tokens [max(0, P + 1 - window) (0 for window 0), P + 1) of KV
 * head g / (n_q / n_kv).  Rows with L <= 0 produce zeros; 0 < L < q_len is
 * an error.  out is double. */
int oracle_decode_attention_mq(int dtype, int num_rows, int q_len, int n_q, int n_kv, int D,
                               const float *q, const void *k_data, const void *v_data,
                               const uint16_t *k_scales, const uint16_t *v_scales,
                               const int32_t *block_table, int bt_stride,
                               const int32_t *seq_lens, int num_pages, double scale, int window,
                               double *out) {
    if (n_kv <= 0 || n_q % n_kv || D % ORACLE_QBLOCK || window < 0 || q_len < 1)
        return ORACLE_BAD_ARG;
    for (int i = 0; i < num_rows; ++i)
        if (seq_lens[i] > (int64_t)bt_stride * ORACLE_PAGE ||
            (seq_lens[i] > 0 && seq_lens[i] < q_len))
            return ORACLE_BAD_ARG;
    const int group = n_q / n_kv;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t x = 0; x < (int64_t)num_rows * q_len * n_q; ++x) {
        int i = (int)(x / ((int64_t)q_len * n_q));
        int j = (int)((x / n_q) % q_len), g = (int)(x % n_q), h = g / group;
        int L = seq_lens[i];
        double *o = out + x * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (L <= 0) continue;
        int P = L - q_len + j;
        if (attend(dtype, k_data, v_data, k_scales, v_scales, n_kv, D, block_table, bt_stride,
                   num_pages, i, h, q + x * D, scale, window_start(P + 1, window), P + 1,
                   o) != ORACLE_OK) {
#pragma omp atomic write
            status = ORACLE_BAD_PAGE;
        }
    }
    return status;
}

/* Partial attention state of one (row i, query head g) over tokens [t0, t1),
 * in base 2: with s2_t = log2(e) * scale * <q, K_t>,
 *   m2 = max_t s2_t,  l = sum_t 2^(s2_t - m2),  acc = sum_t 2^(s2_t - m2) V_t.
 * These are the quantities a split of the token range produces before the
 * splits are merged; acc is double [D]. */
int oracle_attention_partial(int dtype, int n_q, int n_kv, int D, const float *q_row,
                             const void *k_data, const void *v_data,
                             const uint16_t *k_scales, const uint16_t *v_scales,
                             const int32_t *block_table, int bt_stride, int num_pages, int i,
                             int g, double scale, int t0, int t1, double *m2, double *l,
                             double *acc) {
    if (n_kv <= 0 || n_q % n_kv || t1 <= t0) return ORACLE_BAD_ARG;
    int h = g / (n_q / n_kv);
    double *s = (double *)malloc(sizeof(double) * (size_t)(t1 - t0));
    if (!s) return ORACLE_BAD_ARG;
    int st = scores(dtype, k_data, k_scales, n_kv, D, block_table, bt_stride, num_pages, i, h,
                    q_row + (int64_t)g * D, scale, t0, t1, s);
    if (st != ORACLE_OK) { free(s); return st; }
    double m = -INFINITY;
    for (int t = 0; t < t1 - t0; ++t) {
        s[t] *= M_LOG2E;
        m = s[t] > m ? s[t] : m;
    }
    *m2 = m;
    *l = 0.0;
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    for (int t = t0; t < t1; ++t) {
        double p = exp2(s[t - t0] - m);
        *l += p;
        int64_t page = page_of(block_table, bt_stride, i, t, num_pages);
        for (int d = 0; d < D; ++d)
            acc[d] += p * stored(dtype, v_data, v_scales, n_kv, D, page, h, t % ORACLE_PAGE, d);
    }
    free(s);
    return ORACLE_OK;
}

/* Merge n base-2 partial states (m2[s], l[s], acc[s][D]) of disjoint token
 * ranges of one (row, query head) into the attention output:
 *   M = max_s m2[s],  w_s = 2^(m2[s] - M),
 *   out = sum_s w_s acc[s] / sum_s w_s l[s].
 * The inputs are fp32 as the device stores them; the merge runs in double. */
void oracle_combine(int n, const float *m2, const float *l, const float *acc, int D,
                    double *out) {
    double M = -INFINITY;
    for (int s = 0; s < n; ++s) M = m2[s] > M ? m2[s] : M;
    double den = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int s = 0; s < n; ++s) {
        double w = exp2((double)m2[s] - M);
        den += w * (double)l[s];
        for (int d = 0; d < D; ++d) out[d] += w * (double)acc[(int64_t)s * D + d];
    }
    for (int d = 0; d < D; ++d) out[d] /= den;
}

/* --------------------------------------------------------------- plan --- */

/* The work split of one decode call, written out by brute force.
 *
 * Work unit: one (page, KV head) tile of a row.  Row i reads npg_i pages:
 * those that hold a token of [a_i, L_i), a_i = max(0, L_i - window) (a_i = 0
 * for window 0), so npg_i = ceil(L_i / 16) - floor(a_i / 16), 0 for L_i <= 0;
 * its page p < npg_i is block-table entry floor(a_i / 16) + p.  Units are numbered in the order
 * (row, KV head, page): segment j = i * n_kv + h holds the npg_i units of
 * (row i, head h) starting at seg_start(j) = n_kv * sum_{r<i} npg_r + h * npg_i.
 * With T = n_kv * sum_i npg_i units and C chunks requested, the chunks are:
 *   aligned (only when `aligned` is set): walking the rows in order, a row
 *   with npg_i >= t gives, head by head, c = ceil(npg_i / t) chunks of the
 *   head's segment, the q-th holding its pages [floor(q npg_i / c),
 *   floor((q + 1) npg_i / c)); a row with 0 < npg_i < t gives chunks of
 *   m = floor(t / npg_i) consecutive whole segments (the last one what is
 *   left).  t is the first cap, counting up from ceil(T / C) to
 *   floor(11 T / (10 C)), for which this walk makes at most C chunks; if that
 *   range holds a single cap or none, if no cap fits, or if T >= 2^31, the
 *   split is uniform;
 *   uniform: Ce = min(C, T) chunks (so none is empty), chunk k < Ce covering
 *   units [floor(k T / Ce), floor((k + 1) T / Ce)).
 * A segment's pieces are its intersections with the chunks; first/last
 * chunk record which chunks they are (-1, -1 for an empty segment).
 *
 * Outputs: row_page_start[rows + 1] (exclusive prefix sum of npg),
 * seg_first_chunk[rows * n_kv], seg_last_chunk[rows * n_kv], *total = T. */

/* The aligned walk for cap t: the number of chunks it makes, and their unit
 * ranges in lo/hi while they fit in `cap_chunks` entries (lo may be NULL). */
static int64_t aligned_walk(int num_rows, const int32_t *rps, int n_kv, int64_t t,
                            int64_t *lo, int64_t *hi, int64_t cap_chunks) {
    int64_t n = 0;
    for (int i = 0; i < num_rows; ++i) {
        int64_t npg = rps[i + 1] - rps[i], base = (int64_t)n_kv * rps[i];
        if (npg == 0) continue;
        if (npg >= t) {
            int64_t c = (npg + t - 1) / t;
            for (int h = 0; h < n_kv; ++h)
                for (int64_t q = 0; q < c; ++q, ++n)
                    if (lo && n < cap_chunks) {
                        lo[n] = base + h * npg + q * npg / c;
                        hi[n] = base + h * npg + (q + 1) * npg / c;
                    }
        } else {
            int64_t m = t / npg;
            for (int64_t h = 0; h < n_kv; h += m, ++n)
                if (lo && n < cap_chunks) {
                    lo[n] = base + h * npg;
                    hi[n] = base + (h + m < n_kv ? h + m : n_kv) * npg;
                }
        }
    }
    return n;
}

/* The chunks' unit ranges [lo[k], hi[k]) for k < the returned count (at most
 * num_chunks entries are written), for pages per row given by rps. */
static int64_t split_chunks(int num_rows, const int32_t *rps, int n_kv, int num_chunks,
                            int aligned, int64_t *lo, int64_t *hi) {
    int64_t T = (int64_t)n_kv * rps[num_rows];
    if (aligned && T > 0 && T < ((int64_t)1 << 31)) {
        int64_t t0 = (T + num_chunks - 1) / num_chunks, t1 = 11 * T / (10 * (int64_t)num_chunks);
        for (int64_t t = t0; t1 > t0 && t <= t1; ++t)
            if (aligned_walk(num_rows, rps, n_kv, t, NULL, NULL, 0) <= num_chunks)
                return aligned_walk(num_rows, rps, n_kv, t, lo, hi, num_chunks);
    }
    int64_t nch = T < num_chunks ? T : num_chunks;
    for (int64_t k = 0; k < nch; ++k) {
        lo[k] = k * T / nch;
        hi[k] = (k + 1) * T / nch;
    }
    return nch;
}

static void page_counts(int num_rows, const int32_t *seq_lens, int window, int32_t *rps) {
    rps[0] = 0;
    for (int i = 0; i < num_rows; ++i) {
        int L = seq_lens[i] > 0 ? seq_lens[i] : 0;
        int npg = L > 0 ? (L + ORACLE_PAGE - 1) / ORACLE_PAGE - window_start(L, window) / ORACLE_PAGE
                        : 0;
        rps[i + 1] = rps[i] + npg;
    }
}

/* The chunk ranges of the split oracle_plan describes: lo/hi [num_chunks],
 * *used = the chunks holding units. */
int oracle_chunk_ranges(int num_rows, const int32_t *seq_lens, int n_kv, int num_chunks,
                        int window, int aligned, int64_t *lo, int64_t *hi, int64_t *used) {
    if (num_rows < 0 || n_kv <= 0 || num_chunks <= 0 || window < 0) return ORACLE_BAD_ARG;
    int32_t *rps = malloc(sizeof(int32_t) * ((size_t)num_rows + 1));
    if (!rps) return ORACLE_BAD_ARG;
    page_counts(num_rows, seq_lens, window, rps);
    *used = split_chunks(num_rows, rps, n_kv, num_chunks, aligned, lo, hi);
    free(rps);
    return ORACLE_OK;
}

int oracle_plan(int num_rows, const int32_t *seq_lens, int n_kv, int num_chunks, int window,
                int aligned, int32_t *row_page_start, int32_t *seg_first_chunk,
                int32_t *seg_last_chunk, int64_t *total) {
    if (num_rows < 0 || n_kv <= 0 || num_chunks <= 0 || window < 0) return ORACLE_BAD_ARG;
    page_counts(num_rows, seq_lens, window, row_page_start);
    int64_t T = (int64_t)n_kv * row_page_start[num_rows];
    *total = T;
    /* the chunks' unit ranges */
    int64_t *lo = malloc(sizeof(int64_t) * (size_t)num_chunks);
    int64_t *hi = malloc(sizeof(int64_t) * (size_t)num_chunks);
    if (!lo || !hi) {
        free(lo);
        free(hi);
        return ORACLE_BAD_ARG;
    }
    const int64_t nch = split_chunks(num_rows, row_page_start, n_kv, num_chunks, aligned, lo, hi);
    for (int i = 0; i < num_rows; ++i) {
        int64_t npg = row_page_start[i + 1] - row_page_start[i];
        for (int h = 0; h < n_kv; ++h) {
            int64_t j = (int64_t)i * n_kv + h;
            int64_t a = (int64_t)n_kv * row_page_start[i] + h * npg, b = a + npg;
            int32_t first = -1, last = -1;
            for (int64_t k = 0; k < nch; ++k) {
                if (a < b && lo[k] < hi[k] && lo[k] < b && a < hi[k]) { /* non-empty overlap */
                    if (first < 0) first = (int32_t)k;
                    last = (int32_t)k;
                }
            }
            seg_first_chunk[j] = first;
            seg_last_chunk[j] = last;
        }
    }
    free(lo);
    free(hi);
    return ORACLE_OK;
}
