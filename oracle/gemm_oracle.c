/*
 * gemm_oracle.c -- plain, slow, obviously correct CPU oracle for
 *     C[M,N] = epi( A[M,K] . B[N,K]^T )
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header, table or constant with
 * the CUDA library.
 *
 * What it follows:
 *  - Problem statement: TileLang tutorial, chapter 11, "pipelined_gemm.py",
 *    kernel matmul_auto: A is (M, K), B is (N, K), C is (M, N) and the tile
 *    product is T.gemm(A_shared, B_shared, C_local, transpose_B=True) with a
 *    float32 accumulator and a float16 output.  The oracle keeps the plain
 *    definition C[i,j] = sum_k A[i,k] * B[j,k] and accumulates in fp64, which
 *    is exact for every product of two fp16/bf16 values and leaves only a
 *    ~1e-12 relative sum error at K <= 8192.
 *  - ReLU epilogue: max(x, 0), the accumulator clamp of the Triton lecture
 *    notes' matmul example (matmul_relu_kernel); zero and negative sums give
 *    +0.
 *  - Bias: no page defines one.  Reading: a Linear layer's per-output-column
 *    bias (the GELU workload is such a layer, Y = gelu(X . W^T)), one value
 *    per column j in the input format, added to the exact sum before the
 *    epilogue: C[i,j] = epi(sum_k A[i,k] B[j,k] + bias[j]).
 *  - Epilogue: the tanh-approximate GELU, 0.5 x (1 + tanh(sqrt(2/pi) (x +
 *    0.044715 x^3))), as the Triton lecture notes ("GeLU" example) and the
 *    XLA:GPU emitters page (loop-emitter example, function @gelu) write it;
 *    the constant sqrt(2/pi) is taken as 0.7978845608.  Evaluated in fp64
 *    with the C library tanh, applied once to the fp64 sum.
 *  - Output rounding: one round-to-nearest-even from the exact value to the
 *    output type (IEEE 754 binary16 / bfloat16), written here from the
 *    definition of the formats.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no -ffast-math,
 * so every sum is a plain left-to-right fp64 sum).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F16 0
#define ORACLE_BF16 1

/* ---- format decoding (IEEE 754-2008 binary16; bfloat16 = top half of binary32) ---- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t h) {
  const unsigned sign = (unsigned)(h >> 15) & 1u;
  const unsigned expo = (unsigned)(h >> 10) & 0x1fu;
  const unsigned frac = (unsigned)h & 0x3ffu;
  double v;
  if (expo == 0u) {
    v = ldexp((double)frac, -24);                     /* subnormal: frac * 2^-24 */
  } else if (expo == 31u) {
    v = frac ? NAN : INFINITY;
  } else {
    v = ldexp((double)(frac | 0x400u), (int)expo - 25); /* 1.frac * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_double(uint16_t b) {
  const unsigned sign = (unsigned)(b >> 15) & 1u;
  const unsigned expo = (unsigned)(b >> 7) & 0xffu;
  const unsigned frac = (unsigned)b & 0x7fu;
  double v;
  if (expo == 0u) {
    v = ldexp((double)frac, -133);                    /* subnormal: frac * 2^(-126-7) */
  } else if (expo == 255u) {
    v = frac ? NAN : INFINITY;
  } else {
    v = ldexp((double)(frac | 0x80u), (int)expo - 134); /* 1.frac * 2^(e-127) */
  }
  return sign ? -v : v;
}

double oracle_decode(uint16_t bits, int dtype) {
  return dtype == ORACLE_BF16 ? oracle_bf16_to_double(bits) : oracle_f16_to_double(bits);
}

/* ---- round to nearest, ties to even, from a double -------------------------
 * Generic over the format: `mant_bits` fraction bits, smallest normal
 * exponent `emin`, largest finite value `max_finite`.  The quantum of the
 * binade that holds |x| is 2^(floor(log2|x|) - mant_bits) for normal values
 * and 2^(emin - mant_bits) below the normal range; nearbyint() rounds the
 * scaled value ties-to-even (default FE_TONEAREST mode).  Results above the
 * largest finite value overflow to infinity, as IEEE round-to-nearest does. */
static uint16_t round_generic(double x, int mant_bits, int emin, int exp_bits) {
  const int bias = (1 << (exp_bits - 1)) - 1;
  const uint16_t inf_bits = (uint16_t)(((1u << exp_bits) - 1u) << mant_bits);
  const uint16_t sign = signbit(x) ? (uint16_t)0x8000u : (uint16_t)0u;
  if (isnan(x)) return (uint16_t)(inf_bits | (1u << (mant_bits - 1)));
  double a = fabs(x);
  if (isinf(a)) return (uint16_t)(sign | inf_bits);
  if (a == 0.0) return sign;
  int e2;
  (void)frexp(a, &e2);               /* a = f * 2^e2, f in [0.5, 1) */
  const int floor_log2 = e2 - 1;
  const int q = (floor_log2 >= emin) ? (floor_log2 - mant_bits) : (emin - mant_bits);
  const double r = nearbyint(ldexp(a, -q)); /* exact scaling by a power of two */
  const double v = ldexp(r, q);
  const double max_finite = ldexp((double)((1u << (mant_bits + 1)) - 1u), bias - mant_bits);
  if (v > max_finite) return (uint16_t)(sign | inf_bits);
  if (v == 0.0) return sign;
  if (v < ldexp(1.0, emin)) {        /* subnormal: count of 2^(emin-mant_bits) */
    return (uint16_t)(sign | (uint16_t)ldexp(v, mant_bits - emin));
  }
  int ev;
  const double f = frexp(v, &ev);    /* v = f * 2^ev, f in [0.5, 1) */
  const unsigned biased = (unsigned)(ev - 1 + bias);
  const unsigned frac = (unsigned)ldexp(f, mant_bits + 1) - (1u << mant_bits);
  return (uint16_t)(sign | (biased << mant_bits) | frac);
}

uint16_t oracle_double_to_f16(double x) { return round_generic(x, 10, -14, 5); }
uint16_t oracle_double_to_bf16(double x) { return round_generic(x, 7, -126, 8); }

/* ---- ReLU ---- */
double oracle_relu(double x) { return x > 0.0 ? x : 0.0; }

/* ---- tanh-GELU ---- */
double oracle_gelu_tanh(double x) {
  const double c = 0.7978845608; /* sqrt(2/pi) */
  return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
}

/* Epilogue selector: 0 none, 1 tanh-GELU, 2 ReLU. */
static double apply_epilogue(double s, int epilogue) {
  if (epilogue == 1) return oracle_gelu_tanh(s);
  if (epilogue == 2) return oracle_relu(s);
  return s;
}

static void set_threads(int threads) {
#ifdef _OPENMP
  if (threads > 0) omp_set_num_threads(threads);
#else
  (void)threads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Decode a whole row-major matrix of 16-bit patterns to doubles. */
static double* decode_matrix(const uint16_t* bits, int64_t count, int dtype) {
  double* out = (double*)malloc((size_t)(count > 0 ? count : 1) * sizeof(double));
  if (!out) return NULL;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) out[i] = oracle_decode(bits[i], dtype);
  return out;
}

/* Bias of output column j: its exact value, or 0 without a bias vector. */
static double bias_of(const uint16_t* bias, int64_t j, int dtype) {
  return bias ? oracle_decode(bias[j], dtype) : 0.0;
}

/* C[i,j] = epi(sum_k A[i,k] * B[j,k] + bias[j]), all in fp64; epilogue 0
 * none, 1 tanh-GELU, 2 ReLU; bias: N values in the input format, or NULL.
 * A: M x K row-major, B: N x K row-major, C: M x N row-major doubles.
 * Returns 0 on success, -1 on bad arguments or allocation failure. */
int oracle_gemm_nt_bias(const uint16_t* A, const uint16_t* B, const uint16_t* bias, int64_t M,
                        int64_t N, int64_t K, int dtype, int epilogue, double* C, int threads) {
  if (M < 0 || N < 0 || K < 0 || !C) return -1;
  if ((M > 0 && K > 0 && !A) || (N > 0 && K > 0 && !B)) return -1;
  set_threads(threads);
  double* Ad = decode_matrix(A, M * K, dtype);
  double* Bd = decode_matrix(B, N * K, dtype);
  if (!Ad || !Bd) { free(Ad); free(Bd); return -1; }
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < M; ++i) {
    const double* a = Ad + i * K;
    for (int64_t j = 0; j < N; ++j) {
      const double* b = Bd + j * K;
      double s = 0.0;
      for (int64_t k = 0; k < K; ++k) s += a[k] * b[k];
      C[i * N + j] = apply_epilogue(s + bias_of(bias, j, dtype), epilogue);
    }
  }
  free(Ad);
  free(Bd);
  return 0;
}

int oracle_gemm_nt(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N, int64_t K,
                   int dtype, int epilogue, double* C, int threads) {
  return oracle_gemm_nt_bias(A, B, NULL, M, N, K, dtype, epilogue, C, threads);
}

/* Same definition, for `count` chosen entries (rows[t], cols[t]) only, so a
 * full-size product can be checked at sampled positions. */
int oracle_gemm_nt_entries_bias(const uint16_t* A, const uint16_t* B, const uint16_t* bias,
                                int64_t M, int64_t N, int64_t K, int dtype, int epilogue,
                                const int64_t* rows, const int64_t* cols, int64_t count,
                                double* out, int threads) {
  if (M < 0 || N < 0 || K < 0 || count < 0 || (count > 0 && (!rows || !cols || !out))) return -1;
  for (int64_t t = 0; t < count; ++t)
    if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
  set_threads(threads);
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t t = 0; t < count; ++t) {
    const uint16_t* a = A + rows[t] * K;
    const uint16_t* b = B + cols[t] * K;
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k) s += oracle_decode(a[k], dtype) * oracle_decode(b[k], dtype);
    out[t] = apply_epilogue(s + bias_of(bias, cols[t], dtype), epilogue);
  }
  return 0;
}

int oracle_gemm_nt_entries(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N, int64_t K,
                           int dtype, int epilogue, const int64_t* rows, const int64_t* cols,
                           int64_t count, double* out, int threads) {
  return oracle_gemm_nt_entries_bias(A, B, NULL, M, N, K, dtype, epilogue, rows, cols, count, out,
                                     threads);
}

/* Element-wise helpers over arrays, for the Python wrapper. */
void oracle_decode_array(const uint16_t* bits, int64_t n, int dtype, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_decode(bits[i], dtype);
}

void oracle_round_array(const double* x, int64_t n, int dtype, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i)
    out[i] = dtype == ORACLE_BF16 ? oracle_double_to_bf16(x[i]) : oracle_double_to_f16(x[i]);
}

void oracle_gelu_array(const double* x, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_gelu_tanh(x[i]);
}
