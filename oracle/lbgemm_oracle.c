/*
 * lbgemm_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU restatement of the low-bit integer
 * GEMM that the library computes on the GPU.  Only the test suite, the smoke
 * check and the CPU-baseline leg of the benchmark may load this file's
 * shared object; the library's product path never does, and shares no code,
 * header or table with it.
 *
 * Source of the method (cited below as [LBG]):
 *   "Leveraging Large-Scale Data for Efficient Low-Bit CUTLASS GEMM
 *    Optimization via Neural Networks", IEEE Transactions on Big Data --
 *   press summary page.  Intro: the method targets 1-, 4- and 8-bit GEMM;
 *   section 1 ("customizable CUTLASS GEMM templates"): the product is
 *   A x B = C, each output tile accumulating along K.
 *
 * Readings where the page is silent (it gives no layout, packing or 1-bit
 * semantics):
 *   - A is M x K and B is N x K, both K-major; C[m][n] = sum_k A[m][k]*B[n][k]
 *     (C = A * B^T), C row-major int32.
 *   - 8-bit: signed two's complement, full range [-128, 127].
 *   - 4-bit: signed nibbles, value = ((nibble ^ 8) - 8); element k of a row
 *     sits in byte k/2, low nibble for even k.  Rows hold ceil(K/2) bytes.
 *   - 1-bit: element k is bit (k % 32) of 32-bit word k/32; bit 1 means +1,
 *     bit 0 means -1.  Rows hold ceil(K/32) words.  The dot product of two
 *     +-1 rows is (#equal) - (#different) = K - 2*popcount(a XOR b).
 *   - Any K >= 1 is accepted here; bits/nibbles past K in the last word/byte
 *     are padding and ignored.
 *   - Every sum is formed in int64; a result that does not fit int32 makes
 *     the call return ORACLE_OVERFLOW (the library rejects such K up front).
 *   - Linear layer (section 4 names a linear layer; the scale form is the
 *     plainest one): ref[m][n] = (double)acc[m][n] * sx[m] * sw[n], in fp64.
 *
 * Threads split the rows of C; nothing else is blocked, fused or reordered.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_OVERFLOW 1
#define ORACLE_BAD_ARG 2

/* ---- element accessors: the value of element k of one row ---------------- */

/* 4-bit: element k lives in byte k/2, low nibble when k is even. */
static int64_t s4_elem(const uint8_t* row, int64_t k) {
  uint8_t byte = row[k / 2];
  unsigned nib = (k % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
  return (int64_t)((int)(nib ^ 8u) - 8); /* two's complement nibble */
}

/* 1-bit: element k is bit k%32 of word k/32; 1 -> +1, 0 -> -1. */
static int64_t b1_elem(const uint32_t* row, int64_t k) {
  uint32_t bit = (row[k / 32] >> (k % 32)) & 1u;
  return bit ? 1 : -1;
}

/* Portable popcount, written out (no builtins): clear the lowest set bit
 * until none is left. */
static int popcount32(uint32_t x) {
  int c = 0;
  while (x) {
    x &= x - 1u;
    ++c;
  }
  return c;
}

/* ---- one output element per operand kind --------------------------------- */

static int64_t dot_s8(const int8_t* a, const int8_t* b, int64_t K) {
  int64_t s = 0;
  for (int64_t k = 0; k < K; ++k) s += (int64_t)a[k] * (int64_t)b[k];
  return s;
}

static int64_t dot_s4(const uint8_t* a, const uint8_t* b, int64_t K) {
  int64_t s = 0;
  for (int64_t k = 0; k < K; ++k) s += s4_elem(a, k) * s4_elem(b, k);
  return s;
}

/* 1-bit, popcount form: K - 2 * popcount(a XOR b) over the K valid bits. */
static int64_t dot_b1_popc(const uint32_t* a, const uint32_t* b, int64_t K) {
  int64_t words = (K + 31) / 32;
  int64_t diff = 0;
  for (int64_t w = 0; w < words; ++w) {
    uint32_t x = a[w] ^ b[w];
    int64_t valid = K - 32 * w; /* bits of this word inside K */
    if (valid < 32) x &= (1u << valid) - 1u;
    diff += popcount32(x);
  }
  return K - 2 * diff;
}

/* 1-bit, unpacked form: map every bit to +-1 and take the ordinary dot. */
static int64_t dot_b1_unpacked(const uint32_t* a, const uint32_t* b, int64_t K) {
  int64_t s = 0;
  for (int64_t k = 0; k < K; ++k) s += b1_elem(a, k) * b1_elem(b, k);
  return s;
}

/* ---- threaded driver over rows of C -------------------------------------- */

enum { KIND_S8 = 0, KIND_S4 = 1, KIND_B1 = 2, KIND_B1_UNPACKED = 3 };

typedef struct {
  int kind;
  int64_t N, K, row_elems; /* row stride of A and B in units of its element */
  const void* A;
  const void* B;
  int32_t* C;
  int64_t r0, r1;
  int overflow;
} job_t;

static int64_t dot_kind(int kind, const void* A, const void* B, int64_t m, int64_t n,
                        int64_t K, int64_t stride) {
  switch (kind) {
    case KIND_S8:
      return dot_s8((const int8_t*)A + m * stride, (const int8_t*)B + n * stride, K);
    case KIND_S4:
      return dot_s4((const uint8_t*)A + m * stride, (const uint8_t*)B + n * stride, K);
    case KIND_B1:
      return dot_b1_popc((const uint32_t*)A + m * stride, (const uint32_t*)B + n * stride, K);
    default:
      return dot_b1_unpacked((const uint32_t*)A + m * stride, (const uint32_t*)B + n * stride,
                             K);
  }
}

static void* run_rows(void* arg) {
  job_t* j = (job_t*)arg;
  for (int64_t m = j->r0; m < j->r1; ++m) {
    for (int64_t n = 0; n < j->N; ++n) {
      int64_t s = dot_kind(j->kind, j->A, j->B, m, n, j->K, j->row_elems);
      if (s > INT32_MAX || s < INT32_MIN) j->overflow = 1;
      j->C[m * j->N + n] = (int32_t)s;
    }
  }
  return NULL;
}

static int64_t row_elems_of(int kind, int64_t K) {
  if (kind == KIND_S8) return K;
  if (kind == KIND_S4) return (K + 1) / 2;
  return (K + 31) / 32;
}

static int gemm_kind(int kind, int64_t M, int64_t N, int64_t K, const void* A, const void* B,
                     int32_t* C, int nthreads) {
  if (M < 0 || N < 0 || K < 1 || (M > 0 && !A) || (N > 0 && !B) || (M * N > 0 && !C))
    return ORACLE_BAD_ARG;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nthreads > M) nthreads = M > 0 ? (int)M : 1;
  job_t jobs[256];
  pthread_t tids[256];
  int64_t per = M / nthreads, extra = M % nthreads, r = 0;
  for (int t = 0; t < nthreads; ++t) {
    int64_t cnt = per + (t < extra ? 1 : 0);
    jobs[t] = (job_t){kind, N, K, row_elems_of(kind, K), A, B, C, r, r + cnt, 0};
    r += cnt;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&tids[t], NULL, run_rows, &jobs[t]) != 0) break;
    started = t;
  }
  run_rows(&jobs[0]);
  /* rows of threads that failed to start are done here */
  for (int t = started + 1; t < nthreads; ++t) run_rows(&jobs[t]);
  int overflow = jobs[0].overflow;
  for (int t = 1; t <= started; ++t) {
    pthread_join(tids[t], NULL);
    overflow |= jobs[t].overflow;
  }
  for (int t = started + 1; t < nthreads; ++t) overflow |= jobs[t].overflow;
  return overflow ? ORACLE_OVERFLOW : ORACLE_OK;
}

/* ---- exported entry points ------------------------------------------------ */

/* C[M,N] = A[M,K] . B[N,K]^T, signed 8-bit operands, int32 result.  [LBG] s1 */
int oracle_gemm_s8(int64_t M, int64_t N, int64_t K, const int8_t* A, const int8_t* B,
                   int32_t* C, int nthreads) {
  return gemm_kind(KIND_S8, M, N, K, A, B, C, nthreads);
}

/* Same product over signed nibbles packed two per byte, low nibble first. */
int oracle_gemm_s4(int64_t M, int64_t N, int64_t K, const uint8_t* A, const uint8_t* B,
                   int32_t* C, int nthreads) {
  return gemm_kind(KIND_S4, M, N, K, A, B, C, nthreads);
}

/* Same product over +-1 values packed 32 per word: K - 2*popcount(a ^ b). */
int oracle_gemm_b1(int64_t M, int64_t N, int64_t K, const uint32_t* A, const uint32_t* B,
                   int32_t* C, int nthreads) {
  return gemm_kind(KIND_B1, M, N, K, A, B, C, nthreads);
}

/* The 1-bit product again, through the unpacked +-1 values: an independent
 * formulation used to cross-check the popcount form. */
int oracle_gemm_b1_unpacked(int64_t M, int64_t N, int64_t K, const uint32_t* A,
                            const uint32_t* B, int32_t* C, int nthreads) {
  return gemm_kind(KIND_B1_UNPACKED, M, N, K, A, B, C, nthreads);
}

/* Selected entries only: out[i] = C[rows[i], cols[i]].  bits is 8, 4 or 1.
 * Used where the full product is too large for the CPU. */
int oracle_entries(int bits, int64_t M, int64_t N, int64_t K, const void* A, const void* B,
                   int64_t count, const int64_t* rows, const int64_t* cols, int32_t* out) {
  int kind = bits == 8 ? KIND_S8 : bits == 4 ? KIND_S4 : bits == 1 ? KIND_B1 : -1;
  if (kind < 0 || K < 1 || count < 0) return ORACLE_BAD_ARG;
  int64_t stride = row_elems_of(kind, K);
  int overflow = 0;
  for (int64_t i = 0; i < count; ++i) {
    if (rows[i] < 0 || rows[i] >= M || cols[i] < 0 || cols[i] >= N) return ORACLE_BAD_ARG;
    int64_t s = dot_kind(kind, A, B, rows[i], cols[i], K, stride);
    if (s > INT32_MAX || s < INT32_MIN) overflow = 1;
    out[i] = (int32_t)s;
  }
  return overflow ? ORACLE_OVERFLOW : ORACLE_OK;
}

/* Quantised linear layer, fp64 reference: ref[m][n] = acc[m][n] * sx[m] * sw[n]
 * with acc the exact 8-bit product of X[M,K] and W[N,K].  [LBG] s4 */
int oracle_linear(int64_t M, int64_t N, int64_t K, const int8_t* X, const float* sx,
                  const int8_t* W, const float* sw, double* ref, int nthreads) {
  if (M < 0 || N < 0 || K < 1) return ORACLE_BAD_ARG;
  if (M == 0 || N == 0) return ORACLE_OK;
  int32_t* acc = (int32_t*)malloc((size_t)(M * N) * sizeof(int32_t));
  if (!acc) return ORACLE_BAD_ARG;
  int rc = oracle_gemm_s8(M, N, K, X, W, acc, nthreads);
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n)
      ref[m * N + n] = (double)acc[m * N + n] * (double)sx[m] * (double)sw[n];
  free(acc);
  return rc;
}
