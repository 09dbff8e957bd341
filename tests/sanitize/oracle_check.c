/* The CPU oracle under -fsanitize=address,undefined: every format, block size and activation
 * type on small random problems (codes drawn over their whole range, NaN codes included), with
 * and without bias and column subsets, plus the dense GEMV.  Exits 0 and prints "ok" when it
 * ran through; a sanitizer report makes it fail.  (Compiled and run by tests/test_sanitizers.py.) */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

int orc_dequant_rows(int fmt, int bs, int has_zp, long N, long K, const void* W, const void* S,
                     const void* Z, const void* G, long n0, long count, double* out);
int orc_gemv(int fmt, int bf16, int bs, int has_zp, long N, long K, int M, const void* A,
             const void* W, const void* S, const void* Z, const void* G, const void* bias,
             const void* rows, long nrows, void* ybits, void* exact, void* absdot);
int orc_dense_gemv(int bf16, long N, long K, int M, const void* A, const void* B, void* ybits,
                   void* exact, void* absdot);

static uint64_t state = 0x2545F4914F6CDD1Dull;
static uint32_t rnd(void) {
  state ^= state >> 12;
  state ^= state << 25;
  state ^= state >> 27;
  return (uint32_t)((state * 2685821657736338717ull) >> 32);
}

static void fill(unsigned char* p, size_t n) {
  for (size_t i = 0; i < n; ++i) p[i] = (unsigned char)rnd();
}

int main(void) {
  const int fmts[4] = {1, 2, 3, 4};
  const int int_bs[5] = {16, 32, 64, 128, 256};
  int runs = 0;
  for (int it = 0; it < 400; ++it) {
    const int fmt = fmts[rnd() % 4];
    const int bs = fmt == 3 ? 128 : fmt == 4 ? 16 : int_bs[rnd() % 5];
    const int zp = (fmt <= 2) ? (int)(rnd() % 2) : 0;
    const int bf16 = (int)(rnd() % 2);
    const long N = 1 + rnd() % 70, K = 256L * (1 + rnd() % 3);
    const int M = 1 + (int)(rnd() % 5);
    const long nb = K / bs;
    const size_t wbytes = (size_t)N * (size_t)((fmt == 1 || fmt == 4) ? K / 2 : K);
    const size_t sbytes = (size_t)N * (size_t)nb * (fmt == 3 ? 4 : fmt == 4 ? 1 : 2);
    const size_t zbytes = (size_t)N * (size_t)(fmt == 1 ? (nb + 1) / 2 : nb);
    unsigned char* W = malloc(wbytes);
    unsigned char* S = malloc(sbytes);
    unsigned char* Z = malloc(zbytes);
    uint16_t* A = malloc(sizeof(uint16_t) * (size_t)M * (size_t)K);
    uint16_t* bias = malloc(sizeof(uint16_t) * (size_t)N);
    fill(W, wbytes);
    fill(S, sbytes);
    fill(Z, zbytes);
    fill((unsigned char*)A, sizeof(uint16_t) * (size_t)M * (size_t)K);
    fill((unsigned char*)bias, sizeof(uint16_t) * (size_t)N);
    if (fmt == 3) { /* fp32 scales: finite, positive */
      float* f = (float*)S;
      for (size_t i = 0; i < sbytes / 4; ++i) f[i] = (float)(1 + rnd() % 1000) / 4096.0f;
    }
    const float g = 1.0f / 64.0f;
    double* deq = malloc(sizeof(double) * (size_t)N * (size_t)K);
    if (orc_dequant_rows(fmt, bs, zp, N, K, W, S, zp ? Z : NULL, fmt == 4 ? &g : NULL, 0, N, deq) != 0)
      return 2;
    const size_t cols = (size_t)(N > 3 ? N : 3); /* all N columns, or the 3-column subset */
    uint16_t* y = malloc(sizeof(uint16_t) * (size_t)M * cols);
    double* ex = malloc(sizeof(double) * (size_t)M * cols);
    double* ad = malloc(sizeof(double) * (size_t)M * cols);
    const int with_bias = (int)(rnd() % 2);
    if (orc_gemv(fmt, bf16, bs, zp, N, K, M, A, W, S, zp ? Z : NULL, fmt == 4 ? &g : NULL,
                 with_bias ? bias : NULL, NULL, 0, y, ex, ad) != 0)
      return 3;
    int64_t rows[3] = {0, N - 1, N / 2};
    if (orc_gemv(fmt, bf16, bs, zp, N, K, M, A, W, S, zp ? Z : NULL, fmt == 4 ? &g : NULL, NULL,
                 rows, 3, y, ex, ad) != 0)
      return 4;
    free(W), free(S), free(Z), free(A), free(bias), free(deq), free(y), free(ex), free(ad);
    ++runs;
  }
  for (int it = 0; it < 100; ++it) {
    const long N = 1 + rnd() % 50, K = 1 + rnd() % 300;
    const int M = 1 + (int)(rnd() % 8), bf16 = (int)(rnd() % 2);
    uint16_t* A = malloc(sizeof(uint16_t) * (size_t)M * (size_t)K);
    uint16_t* B = malloc(sizeof(uint16_t) * (size_t)K * (size_t)N);
    fill((unsigned char*)A, sizeof(uint16_t) * (size_t)M * (size_t)K);
    fill((unsigned char*)B, sizeof(uint16_t) * (size_t)K * (size_t)N);
    uint16_t* y = malloc(sizeof(uint16_t) * (size_t)M * (size_t)N);
    double* ex = malloc(sizeof(double) * (size_t)M * (size_t)N);
    double* ad = malloc(sizeof(double) * (size_t)M * (size_t)N);
    if (orc_dense_gemv(bf16, N, K, M, A, B, y, ex, ad) != 0) return 5;
    free(A), free(B), free(y), free(ex), free(ad);
    ++runs;
  }
  printf("ok: %d oracle runs\n", runs);
  return 0;
}
