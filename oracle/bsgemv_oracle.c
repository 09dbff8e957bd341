/*
 * bsgemv_oracle.c -- plain CPU reference ("oracle") for the block-scaled small-M GEMV
 *
 *     y[M, N] = A[M, K] . deq(W)[N, K]^T
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct definition that the CUDA
 * path is checked against.  Only the test suite, the smoke check and the benchmark's CPU
 * baseline / reference arm may load it.  It shares no code, header, table or constant with the
 * CUDA library and includes nothing from it.
 *
 * Everything is computed in IEEE binary64:
 *   1. every stored code (fp16 / bf16 activations and scales, E4M3, E2M1) is decoded to its exact
 *      value by one parametric minifloat decoder written from the formats' definitions;
 *   2. the dequantised weight is formed exactly: (q - zp) * s, e4m3 * s, e2m1 * e4m3 * g -- every
 *      one of these products has at most 4 + 24 significand bits, so binary64 holds it exactly;
 *   3. the dot product over K is summed in increasing k order in binary64;
 *   4. an optional bias[n] (activation dtype, one value per output column) is added to the sum
 *      in binary64;
 *   5. the result is rounded once, round-to-nearest-even, to the activation dtype.
 *
 * Sources (web pages on the method; cited by title and section):
 *   [P1] "[CUDA] Block-scaled MatMul decode GEMV: tensor cores, packed FP4 decode and M-tiling"
 *        (onnxruntime PR #31155), description: the FP8 tensor-core paragraph (E4M3 -> FP16/BF16
 *        lossless, fp32 accumulate) and the NVFP4 tensor-core paragraph (E2M1 x E4M3 block scale,
 *        2 + 4 significand bits, range 2^-10 .. 2688).
 *   [P3] "[CUDA] MatMulNBits 8-bit: wide fp16 M=1 kernel for decode GEMVs" (PR #33728),
 *        Description: exact (q - zp), fp32 accumulation, per-block scale.
 *   [P5] "[CUDA] Batched small-M GEMV for MatMulNBits (4-bit/8-bit)" (PR #29451), Description and
 *        review: the standard [N, blocks, blob] weight layout and its packed zero points.
 *
 * Readings where the pages are silent (the plainest reading consistent with the rest of them):
 *   - int4 packing: two codes per byte, the LOW nibble holds the even k.
 *   - int4 zero points: [N, ceil(nb/2)] bytes, block b in nibble (b & 1) of byte b >> 1 (low nibble
 *     = even block).  int8 zero points: [N, nb] bytes.
 *   - has_zp == 0 means the implicit zero point 2^(bits-1): 8 for int4, 128 for int8.
 *   - int4/int8 scales are fp16 for both activation dtypes; FP8 scales are fp32, one per 128 k;
 *     NVFP4 scales are E4M3 codes, one per 16 k, row-major [N, K/16]; the NVFP4 global scale is one
 *     fp32 number.
 *   - NVFP4 codes are packed like int4 (low nibble = even k).
 *   - The output is rounded round-to-nearest-even; overflow goes to +-inf, NaN propagates.
 *   - Bias: the FP8 / FP4 operators' tests cover an optional bias ([P1] Tests; "[CUDA] Pin FP8 GEMV
 *     residency ...", Tests); read as y = A . deq(W)^T + bias with bias [N] in the activation
 *     dtype, broadcast over the M rows and added before the one rounding.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_INT4 = 1, ORC_INT8 = 2, ORC_FP8_E4M3 = 3, ORC_NVFP4 = 4 };

/* How the all-ones exponent is used by a minifloat format. */
enum {
  ORC_SPECIAL_NONE = 0,   /* E2M1: every code is finite */
  ORC_SPECIAL_FN = 1,     /* E4M3 ("fn"): only S.1111.111 is NaN, no infinities */
  ORC_SPECIAL_IEEE = 2    /* fp16 / bf16: exponent all ones = inf (mantissa 0) or NaN */
};

/* ------------------------------------------------------------------------------------------ */
/* Minifloat decode: the value of a code with 1 sign bit, `ebits` exponent bits (bias `bias`)   */
/* and `mbits` mantissa bits.  Exponent field 0 is subnormal: m * 2^(1 - bias - mbits).         */
/* Otherwise (2^mbits + m) * 2^(e - bias - mbits).                                              */
/* ------------------------------------------------------------------------------------------ */
double orc_minifloat_value(uint32_t code, int ebits, int mbits, int bias, int special) {
  const uint32_t mmask = (1u << mbits) - 1u;
  const uint32_t emask = (1u << ebits) - 1u;
  const uint32_t m = code & mmask;
  const uint32_t e = (code >> mbits) & emask;
  const int neg = (int)((code >> (mbits + ebits)) & 1u);
  double v;
  if (special == ORC_SPECIAL_IEEE && e == emask) {
    v = (m == 0) ? INFINITY : NAN;
  } else if (special == ORC_SPECIAL_FN && e == emask && m == mmask) {
    v = NAN;
  } else if (e == 0) {
    v = ldexp((double)m, 1 - bias - mbits);
  } else {
    v = ldexp((double)((1u << mbits) + m), (int)e - bias - mbits);
  }
  return neg ? -v : v;
}

double orc_f16_value(uint32_t bits) { return orc_minifloat_value(bits, 5, 10, 15, ORC_SPECIAL_IEEE); }
double orc_bf16_value(uint32_t bits) { return orc_minifloat_value(bits, 8, 7, 127, ORC_SPECIAL_IEEE); }
/* E4M3: 4 exponent bits, bias 7, 3 mantissa bits; max finite 448 (code 0x7E). [P1] */
double orc_e4m3_value(uint32_t code) { return orc_minifloat_value(code, 4, 3, 7, ORC_SPECIAL_FN); }
/* E2M1: 2 exponent bits, bias 1, 1 mantissa bit ("2 significand bits"); max 6. [P1] */
double orc_e2m1_value(uint32_t code) { return orc_minifloat_value(code, 2, 1, 1, ORC_SPECIAL_NONE); }

/* ------------------------------------------------------------------------------------------ */
/* Round a binary64 number to the nearest minifloat code, ties to even.  The quantum (spacing) */
/* at |x| is 2^(exponent of the leading bit - mbits), never below the subnormal spacing.       */
/* Results past the largest finite value become inf (IEEE formats) or saturate to NaN per the  */
/* format (only used with IEEE formats for outputs).                                            */
/* ------------------------------------------------------------------------------------------ */
uint32_t orc_round_minifloat(double x, int ebits, int mbits, int bias, int special) {
  const uint32_t sign = signbit(x) ? (1u << (ebits + mbits)) : 0u;
  const uint32_t emask = (1u << ebits) - 1u;
  if (isnan(x)) {
    /* canonical NaN: exponent all ones with the top mantissa bit (IEEE) or all ones (fn) */
    if (special == ORC_SPECIAL_FN) return (emask << mbits) | ((1u << mbits) - 1u);
    return (emask << mbits) | (1u << (mbits - 1));
  }
  const double a = fabs(x);
  /* largest finite exponent field and mantissa */
  const uint32_t emax_field = (special == ORC_SPECIAL_IEEE) ? emask - 1u : emask;
  const uint32_t mmax = (special == ORC_SPECIAL_FN) ? (1u << mbits) - 2u : (1u << mbits) - 1u;
  if (isinf(a)) {
    return sign | (emask << mbits);
  }
  if (a == 0.0) return sign;

  int fexp;
  (void)frexp(a, &fexp);                  /* a = f * 2^fexp, f in [0.5, 1): leading bit 2^(fexp-1) */
  int qexp = (fexp - 1) - mbits;          /* spacing of the binade that holds a */
  const int qmin = 1 - bias - mbits;      /* subnormal spacing */
  if (qexp < qmin) qexp = qmin;
  const double r = ldexp(a, -qexp);       /* exact: scaling by a power of two */
  double n = floor(r);
  const double frac = r - n;              /* exact */
  if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;
  const double v = ldexp(n, qexp);        /* the rounded magnitude, exact */

  /* encode v */
  const double maxfinite = ldexp((double)((1u << mbits) + mmax), (int)emax_field - bias - mbits);
  if (v > maxfinite) {
    if (special == ORC_SPECIAL_IEEE) return sign | (emask << mbits);
    if (special == ORC_SPECIAL_FN) return sign | (emask << mbits) | ((1u << mbits) - 1u);
    return sign | (emax_field << mbits) | mmax; /* no special values: saturate */
  }
  if (v < ldexp(1.0, 1 - bias)) {         /* subnormal (or the smallest normal after rounding) */
    const uint32_t m = (uint32_t)ldexp(v, -qmin);
    return sign | m;                      /* m == 2^mbits carries into exponent 1 correctly */
  }
  int vexp;
  (void)frexp(v, &vexp);
  const uint32_t e = (uint32_t)((vexp - 1) + bias);
  const uint32_t m = (uint32_t)(ldexp(v, -((vexp - 1) - mbits)) - ldexp(1.0, mbits));
  return sign | (e << mbits) | m;
}

uint32_t orc_round_f16(double x) { return orc_round_minifloat(x, 5, 10, 15, ORC_SPECIAL_IEEE); }
uint32_t orc_round_bf16(double x) { return orc_round_minifloat(x, 8, 7, 127, ORC_SPECIAL_IEEE); }

/* array helpers for the Python wrapper */
void orc_decode_array(const uint32_t* codes, double* out, long n, int ebits, int mbits, int bias,
                      int special) {
  for (long i = 0; i < n; ++i) out[i] = orc_minifloat_value(codes[i], ebits, mbits, bias, special);
}
void orc_round_array(const double* x, uint32_t* out, long n, int ebits, int mbits, int bias,
                     int special) {
  for (long i = 0; i < n; ++i) out[i] = orc_round_minifloat(x[i], ebits, mbits, bias, special);
}

/* ------------------------------------------------------------------------------------------ */
/* Dequantisation of one weight row n, written out per format.                                 */
/* ------------------------------------------------------------------------------------------ */
typedef struct {
  int fmt;          /* ORC_INT4 .. ORC_NVFP4 */
  int block_size;   /* bs: k-elements per scale block */
  int has_zp;       /* int formats only */
  long N, K;
  const uint8_t* W; /* [N, K/bs, blob] bytes */
  const void* scales;
  const uint8_t* zp;
  double gscale;    /* NVFP4 global scale (already decoded from fp32) */
} orc_weights;

/* Row pitch in bytes of the weight: the [N, blocks, blob] layout has blob = bs * bits / 8. [P5] */
static long orc_w_row_bytes(const orc_weights* w) {
  return (w->fmt == ORC_INT4 || w->fmt == ORC_NVFP4) ? w->K / 2 : w->K;
}

/* The code q(n, k) as stored. */
static uint32_t orc_code(const orc_weights* w, long n, long k) {
  const uint8_t* row = w->W + n * orc_w_row_bytes(w);
  if (w->fmt == ORC_INT4 || w->fmt == ORC_NVFP4) {
    const uint8_t byte = row[k / 2];
    return (k % 2 == 0) ? (byte & 0x0Fu) : (byte >> 4);   /* low nibble = even k */
  }
  return row[k];
}

/* Exact dequantised value of W[n, k]. */
static double orc_deq(const orc_weights* w, long n, long k) {
  const long bs = w->block_size;
  const long nb = w->K / bs;
  const long b = k / bs;
  const uint32_t q = orc_code(w, n, k);
  switch (w->fmt) {
    case ORC_INT4: {
      /* deq = (q - zp) * s, s an fp16 per (n, block); zp packed two per byte [P3, P5] */
      const uint16_t* s = (const uint16_t*)w->scales;
      long zp = 8;
      if (w->has_zp) {
        const long zrow = (nb + 1) / 2;
        const uint8_t zbyte = w->zp[n * zrow + b / 2];
        zp = (b % 2 == 0) ? (zbyte & 0x0F) : (zbyte >> 4);
      }
      const long d = (long)q - zp;                   /* exact small integer in [-15, 15] */
      return (double)d * orc_f16_value(s[n * nb + b]);
    }
    case ORC_INT8: {
      const uint16_t* s = (const uint16_t*)w->scales;
      const long zp = w->has_zp ? (long)w->zp[n * nb + b] : 128;
      const long d = (long)q - zp;                   /* exact integer in [-255, 255] */
      return (double)d * orc_f16_value(s[n * nb + b]);
    }
    case ORC_FP8_E4M3: {
      /* deq = e4m3(q) * s, s an fp32 per (n, 128-block) [P1] */
      const float* s = (const float*)w->scales;
      return orc_e4m3_value(q) * (double)s[n * nb + b];
    }
    case ORC_NVFP4: {
      /* deq = e2m1(q) * e4m3(S[n, k/16]) * g [P1] */
      const uint8_t* s = (const uint8_t*)w->scales;
      return orc_e2m1_value(q) * orc_e4m3_value(s[n * nb + b]) * w->gscale;
    }
  }
  return NAN;
}

/* Dequantise rows [n0, n0 + count) into out[count][K]. */
int orc_dequant_rows(int fmt, int block_size, int has_zp, long N, long K, const uint8_t* W,
                     const void* scales, const uint8_t* zp, const float* gscale, long n0,
                     long count, double* out) {
  orc_weights w = {fmt, block_size, has_zp, N, K, W, scales, zp, gscale ? (double)*gscale : 1.0};
  if (block_size <= 0 || K % block_size != 0 || n0 < 0 || n0 + count > N) return -1;
  for (long i = 0; i < count; ++i)
    for (long k = 0; k < K; ++k) out[i * K + k] = orc_deq(&w, n0 + i, k);
  return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* The GEMV: for every requested output column n (rows[] of W, or all n if rows == NULL) and   */
/* every activation row m < M:                                                                  */
/*    exact[m][i]  = sum_k A[m,k] * deq(n,k)     (binary64, increasing k)  [+ bias[n]]          */
/*    absdot[m][i] = sum_k |A[m,k] * deq(n,k)|   (for the tolerance bound) [+ |bias[n]|]        */
/*    ybits[m][i]  = RNE of exact to the activation dtype                                      */
/* A is [M, K] and bias [N] (NULL: no bias) fp16 (act_bf16 == 0) or bf16 (act_bf16 == 1) bit   */
/* patterns.                                                                                    */
/* ------------------------------------------------------------------------------------------ */
int orc_gemv(int fmt, int act_bf16, int block_size, int has_zp, long N, long K, int M,
             const uint16_t* A, const uint8_t* W, const void* scales, const uint8_t* zp,
             const float* gscale, const uint16_t* bias, const long* rows, long nrows,
             uint16_t* ybits, double* exact, double* absdot) {
  if (block_size <= 0 || K % block_size != 0 || M < 1) return -1;
  const long count = rows ? nrows : N;
  orc_weights w = {fmt, block_size, has_zp, N, K, W, scales, zp, gscale ? (double)*gscale : 1.0};

  /* the activations decoded once: a[m][k] */
  double* a = (double*)malloc(sizeof(double) * (size_t)M * (size_t)K);
  if (!a) return -2;
  for (long i = 0; i < (long)M * K; ++i)
    a[i] = act_bf16 ? orc_bf16_value(A[i]) : orc_f16_value(A[i]);

  int bad = 0;
#pragma omp parallel for schedule(dynamic, 8)
  for (long i = 0; i < count; ++i) {
    const long n = rows ? rows[i] : i;
    if (n < 0 || n >= N) { bad = 1; continue; }
    for (int m = 0; m < M; ++m) {
      double sum = 0.0, asum = 0.0;
      const double* am = a + (long)m * K;
      for (long k = 0; k < K; ++k) {
        const double p = am[k] * orc_deq(&w, n, k);
        sum += p;
        asum += fabs(p);
      }
      if (bias) {
        const double b = act_bf16 ? orc_bf16_value(bias[n]) : orc_f16_value(bias[n]);
        sum += b;
        asum += fabs(b);
      }
      if (exact) exact[(long)m * count + i] = sum;
      if (absdot) absdot[(long)m * count + i] = asum;
      if (ybits) ybits[(long)m * count + i] = (uint16_t)(act_bf16 ? orc_round_bf16(sum)
                                                                  : orc_round_f16(sum));
    }
  }
  free(a);
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Dense GEMV ("[CUDA] MatMul: add an opt-in split-K GEMV for small-N fp16 shapes",          */
/* Description): y[m][n] = sum_k A[m,k] * B[k,n] with A [M, K] and B [K, N] row-major fp16     */
/* (act_bf16 == 0) or bf16 bit patterns; every product is exact in binary64, the sum runs in   */
/* increasing k, the result is rounded once (RNE) to the same dtype.  absdot as orc_gemv.      */
/* ------------------------------------------------------------------------------------------ */
int orc_dense_gemv(int act_bf16, long N, long K, int M, const uint16_t* A, const uint16_t* B,
                   uint16_t* ybits, double* exact, double* absdot) {
  if (N < 1 || K < 1 || M < 1) return -1;
#pragma omp parallel for schedule(static)
  for (long n = 0; n < N; ++n) {
    for (int m = 0; m < M; ++m) {
      double sum = 0.0, asum = 0.0;
      for (long k = 0; k < K; ++k) {
        const uint16_t a = A[(long)m * K + k], b = B[k * N + n];
        const double p = act_bf16 ? orc_bf16_value(a) * orc_bf16_value(b)
                                  : orc_f16_value(a) * orc_f16_value(b);
        sum += p;
        asum += fabs(p);
      }
      if (exact) exact[(long)m * N + n] = sum;
      if (absdot) absdot[(long)m * N + n] = asum;
      if (ybits) ybits[(long)m * N + n] = (uint16_t)(act_bf16 ? orc_round_bf16(sum)
                                                              : orc_round_f16(sum));
    }
  }
  return 0;
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
