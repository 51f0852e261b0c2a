/*
 * CPU oracle for the NVFP4 weight-only skinny projection  y = x . dequant(W)^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * bench's CPU-baseline leg may load this library.  It shares no code, table
 * or header with the CUDA path and must never be used to produce a product
 * result.
 *
 * Everything is computed in IEEE binary64, element by element, with the sum
 * over k taken in ascending k.  There is no blocking, no fusion and no table:
 * each format is decoded from its bit fields by its closed form.
 *
 * Sources (web pages; section / entry named):
 *   [P1] "10 Kernels", section 10.2 "NVFP4 matrix products": the weight is
 *        4-bit E2M1 with an E4M3 group scale multiplied onto it; activations
 *        are 16-bit; one E4M3 scale per 16-element group along K.
 *   [P3] "Module ops" (rustdoc API index), Functions:
 *        - dequant_nvfp4_to_bf16: W[n,k] is packed E2M1 times the E4M3 group
 *          scale times the per-tensor scale2;
 *        - nvfp4_mmq_repack: codes are E2M1 [n, k/2] bytes, LOW nibble = EVEN
 *          k; scales are E4M3 [n, k/16];
 *        - w4a16_gemm: the per-tensor scale is FP32; A is BF16 [M, K];
 *        - w4a16_tc_rows: output[m, n] = input[m, :] . W[n, :]^T for the
 *          row-major NVFP4 weight [n, k].
 *        Constants: E4M3_MAX = E4M3's largest finite magnitude (448).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - E2M1 value set: the OCP Microscaling (MX) v1.0 FP4 E2M1 definition
 *     (sign bit 3, exponent bits 2..1 with bias 1, mantissa bit 0, exponent 0
 *     is subnormal, no Inf/NaN).
 *   - E4M3: the OCP FP8 E4M3FN definition (bias 7, exponent 0 subnormal,
 *     S.1111.111 is NaN, no Inf), which is the one whose largest finite value
 *     is 448 as the pages state.
 *   - The per-tensor scale multiplies each weight element; in binary64 this
 *     is the same value as multiplying the finished sum.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* E2M1 value of a 4-bit code (OCP MX FP4: s | e1 e0 | m, bias 1). */
double nvfp4_oracle_e2m1(unsigned code) {
  unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
  double mag;
  if (e == 0) mag = ldexp((double)m, -1);                     /* subnormal: m/2 * 2^(1-1) */
  else mag = ldexp(1.0 + (double)m / 2.0, (int)e - 1);        /* normal: 1.m * 2^(e-1)    */
  return s ? -mag : mag;
}

/* E4M3 value of one byte (OCP FP8 E4M3FN: s | eeee | mmm, bias 7). */
double nvfp4_oracle_e4m3(unsigned byte) {
  unsigned s = (byte >> 7) & 1u, e = (byte >> 3) & 15u, m = byte & 7u;
  double mag;
  if (e == 15u && m == 7u) return NAN;                        /* the only NaN encodings */
  if (e == 0) mag = ldexp((double)m / 8.0, 1 - 7);            /* subnormal: 0.mmm * 2^-6 */
  else mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);        /* normal: 1.mmm * 2^(e-7) */
  return s ? -mag : mag;
}

/* bfloat16 value of a 16-bit pattern (s | 8 exponent bits, bias 127 | 7 mantissa bits). */
double nvfp4_oracle_bf16(unsigned bits) {
  unsigned s = (bits >> 15) & 1u, e = (bits >> 7) & 255u, m = bits & 127u;
  double mag;
  if (e == 255u) mag = m ? NAN : INFINITY;
  else if (e == 0) mag = ldexp((double)m / 128.0, 1 - 127);
  else mag = ldexp(1.0 + (double)m / 128.0, (int)e - 127);
  return s ? -mag : mag;
}

/* E2M1 code of weight element (n, k): byte n*K/2 + k/2, low nibble for even k. */
static unsigned code_at(const uint8_t* codes, int64_t K, int64_t n, int64_t k) {
  uint8_t b = codes[n * (K / 2) + k / 2];
  return (k & 1) ? (unsigned)(b >> 4) : (unsigned)(b & 15u);
}

/* Dequantised weight element W[n,k] = E2M1(code) * E4M3(scale[n, k/16]) * gs. */
double nvfp4_oracle_weight(const uint8_t* codes, const uint8_t* scales, float gs,
                           int64_t K, int64_t n, int64_t k) {
  double v = nvfp4_oracle_e2m1(code_at(codes, K, n, k));
  double s = nvfp4_oracle_e4m3(scales[n * (K / 16) + k / 16]);
  return v * s * (double)gs;
}

/* One output: y[m,n] = sum_k W[n,k] * x[m,k], and absdot = sum_k |W[n,k] * x[m,k]|. */
static void one_output(int64_t K, const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                       float gs, int64_t m, int64_t n, double* y, double* absdot) {
  double acc = 0.0, aacc = 0.0;
  for (int64_t k = 0; k < K; ++k) {
    double t = nvfp4_oracle_weight(codes, scales, gs, K, n, k) * nvfp4_oracle_bf16(x[m * K + k]);
    acc += t;
    aacc += fabs(t);
  }
  *y = acc;
  *absdot = aacc;
}

/* Full product: y[M,N], absdot[M,N] (row-major, binary64).  nthreads <= 0: library default. */
void nvfp4_oracle_linear(int64_t M, int64_t N, int64_t K, const uint16_t* x, const uint8_t* codes,
                         const uint8_t* scales, float gs, double* y, double* absdot, int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
  for (int64_t n = 0; n < N; ++n)
    for (int64_t m = 0; m < M; ++m)
      one_output(K, x, codes, scales, gs, m, n, &y[m * N + n], &absdot[m * N + n]);
  (void)nthreads;
}

/* Sampled outputs: for i < count, (ms[i], ns[i]) -> y[i], absdot[i]. */
void nvfp4_oracle_linear_at(int64_t K, int64_t count, const int64_t* ms, const int64_t* ns,
                            const uint16_t* x, const uint8_t* codes, const uint8_t* scales, float gs,
                            double* y, double* absdot, int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
  for (int64_t i = 0; i < count; ++i)
    one_output(K, x, codes, scales, gs, ms[i], ns[i], &y[i], &absdot[i]);
  (void)nthreads;
}

/* One bfloat16 ulp at magnitude |a|: 2^(floor(log2|a|) - 7) for normal range, 2^-133 below it. */
double nvfp4_oracle_bf16_ulp(double a) {
  a = fabs(a);
  if (!(a >= ldexp(1.0, -126))) return ldexp(1.0, -133);
  int e;
  frexp(a, &e);               /* a = f * 2^e, f in [0.5, 1): floor(log2 a) = e - 1 */
  return ldexp(1.0, e - 1 - 7);
}

/* Threads the OpenMP runtime would use (1 without OpenMP). */
int nvfp4_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
