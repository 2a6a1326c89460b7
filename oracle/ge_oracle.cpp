// ge_oracle.cpp -- plain CPU oracle for the fused linear-layer path.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or
// load this file: only the tests, the smoke check and the CPU-baseline leg
// of the benchmark do. It shares no code, header, table or constant with the
// CUDA library; the two are compared on identical fp16 bit patterns.
//
// What it computes is the plain definition of the fused epilogue GEMM, in
// fp64, with no blocking, fusion or reordering:
//
//   z[m,n] = sum_k A[m,k] * B[k,n]  (k ascending, fp64)          -- the GEMM
//          + bias[m]                (broadcast over every column) -- BIAS
//   y[m,n] = act(z[m,n])            NONE | ReLU | tanh-GELU | erf-GELU
//   D[m,n] = fp16(y[m,n])           round to nearest even         -- one store
//            (or bfloat16: the *_dt entry points take the element type)
//   mask   = (z > 0) bit-packed     (RELU_AUX_BIAS only)          -- aux output
//
// Sources (page title, section):
//  * nvmath-python cuBLASLt bias-fusion guide, "Core API and parameter
//    configuration": D = weights @ x + bias with bias of shape (m,1) added to
//    every column of the (m,n) product; fp16 inputs and output with a 32-bit
//    compute type ("Advanced techniques", precision item).
//  * same page, "Advanced techniques": RELU_BIAS / GELU_BIAS apply ReLU or GELU
//    to Wx+b; DRELU_BGRAD applies the ReLU gradient mask in the backward pass
//    and accumulates the bias gradient.
//  * Fusing bias addition with matrix multiplication using nvmath-python:
//    Y = ReLU(WX + B); RELU_AUX_BIAS keeps an auxiliary output for backward.
//  * ops-nn MatMul fusion (codearts), "ops-nn's MatMul fusion strategy",
//    first level: the fused and the three-step flows compute the same values.
// Readings where the pages are silent (GELU form = tanh approximation; mask
// bit = z > 0 on the unrounded pre-activation, 32 bits per word along the
// contiguous dimension of stored D, rows padded to 16 bytes; bias gradient =
// sum over tokens of the masked dY) are the plainest ones the pages support.
//
// Pins (tests/test_oracle_pins.py): hand-worked 2x3x4 example, brute-force
// triple loops on tiny inputs in every layout, exhaustive fp16 decode and
// encode against a library conversion, tanh-GELU against an independent
// sigmoid identity and a library GELU, ReLU(z) == z*mask, the exact
// integer-valued case, and the bias gradient against a second summation.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// Epilogue codes of this oracle (its own numbering; the Python wrapper maps
// names to these).
enum OraEpi { ORA_NONE = 0, ORA_BIAS = 1, ORA_RELU_BIAS = 2, ORA_GELU_BIAS = 3,
              ORA_RELU_AUX_BIAS = 4, ORA_GELU_ERF_BIAS = 6, ORA_GELU_AUX_BIAS = 7 };

// IEEE-754 binary16 -> binary64, written from the format definition:
// 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
double f16_decode(uint16_t h) {
  const int s = h >> 15;
  const int e = (h >> 10) & 31;
  const int f = h & 1023;
  double v;
  if (e == 0)
    v = std::ldexp((double)f, -24);             // zero / subnormal: f * 2^-24
  else if (e == 31)
    v = f ? std::nan("") : INFINITY;            // inf / NaN
  else
    v = std::ldexp((double)(1024 + f), e - 25); // (1 + f/1024) * 2^(e-15)
  return s ? -v : v;
}

// Round a non-negative double (< 2^52) to the nearest integer, ties to even.
double round_half_even(double q) {
  const double fl = std::floor(q);
  const double r = q - fl;  // exact for q < 2^52
  if (r > 0.5) return fl + 1.0;
  if (r < 0.5) return fl;
  return std::fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;
}

// binary64 -> binary16 with round-to-nearest-even, overflow to +-inf,
// subnormals kept (no flush to zero).
uint16_t f16_encode(double x) {
  if (std::isnan(x)) return 0x7E00;
  const uint16_t s = std::signbit(x) ? 0x8000 : 0;
  const double a = std::fabs(x);
  // 65504 is the largest finite half; 65520 is the midpoint to 2^16 and ties
  // to the even neighbour, which is the overflow, so it rounds to infinity.
  if (a >= 65520.0) return s | 0x7C00;
  if (a < std::ldexp(1.0, -14)) {
    // subnormal range: value = q * 2^-24, q in [0, 1024]; q == 1024 is the
    // smallest normal, whose bit pattern is also 1024.
    const double q = round_half_even(std::ldexp(a, 24));
    return s | (uint16_t)q;
  }
  int E;
  std::frexp(a, &E);           // a = f * 2^E, f in [0.5, 1)
  int e = E - 1;               // a in [2^e, 2^(e+1))
  double q = round_half_even(std::ldexp(a, 10 - e));  // in [1024, 2048]
  if (q == 2048.0) { q = 1024.0; e += 1; }
  if (e + 15 >= 31) return s | 0x7C00;
  return s | (uint16_t)((e + 15) << 10) | (uint16_t)(q - 1024.0);
}

// bfloat16 -> binary64: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
double bf16_decode(uint16_t h) {
  const int s = h >> 15;
  const int e = (h >> 7) & 255;
  const int f = h & 127;
  double v;
  if (e == 0)
    v = std::ldexp((double)f, -133);             // zero / subnormal: f * 2^-133
  else if (e == 255)
    v = f ? std::nan("") : INFINITY;
  else
    v = std::ldexp((double)(128 + f), e - 134);  // (1 + f/128) * 2^(e-127)
  return s ? -v : v;
}

// binary64 -> bfloat16, round to nearest even, overflow to +-inf, subnormals kept.
uint16_t bf16_encode(double x) {
  if (std::isnan(x)) return 0x7FC0;
  const uint16_t s = std::signbit(x) ? 0x8000 : 0;
  const double a = std::fabs(x);
  // largest finite: (2 - 2^-7) 2^127; the midpoint to 2^128 ties to the
  // even neighbour, which is the overflow.
  if (a >= std::ldexp(511.0, 119)) return s | 0x7F80;  // midpoint (2 - 2^-8) 2^127 = 511 * 2^119
  if (a < std::ldexp(1.0, -126)) {
    const double q = round_half_even(std::ldexp(a, 133));  // units of 2^-133, q <= 128
    return s | (uint16_t)q;
  }
  int E;
  std::frexp(a, &E);
  int e = E - 1;                                        // a in [2^e, 2^(e+1))
  double q = round_half_even(std::ldexp(a, 7 - e));     // in [128, 256]
  if (q == 256.0) { q = 128.0; e += 1; }
  if (e + 127 >= 255) return s | 0x7F80;
  return s | (uint16_t)((e + 127) << 7) | (uint16_t)(q - 128.0);
}

// Element type of the operands, bias and output: 0 = fp16, 1 = bfloat16.
double decode(int dt, uint16_t h) { return dt == 0 ? f16_decode(h) : bf16_decode(h); }
uint16_t encode(int dt, double x) { return dt == 0 ? f16_encode(x) : bf16_encode(x); }

// The activation applied after the bias add.
double activation(int epi, double z) {
  switch (epi) {
    case ORA_RELU_BIAS:
    case ORA_RELU_AUX_BIAS:
      return z > 0.0 ? z : 0.0;
    case ORA_GELU_BIAS:
    case ORA_GELU_AUX_BIAS: {
      // tanh form: 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3)))
      const double c = std::sqrt(2.0 / 3.14159265358979323846);
      return 0.5 * z * (1.0 + std::tanh(c * (z + 0.044715 * z * z * z)));
    }
    case ORA_GELU_ERF_BIAS:
      // exact form: z * Phi(z) = 0.5 z (1 + erf(z / sqrt(2)))
      return 0.5 * z * (1.0 + std::erf(z / std::sqrt(2.0)));
    default:
      return z;
  }
}

// Derivative of the tanh-form GELU with respect to its input, by the product
// and chain rules: with u = c (z + a z^3), t = tanh(u),
//   d/dz [0.5 z (1 + t)] = 0.5 (1 + t) + 0.5 z (1 - t^2) c (1 + 3 a z^2).
double gelu_tanh_grad(double z) {
  const double c = std::sqrt(2.0 / 3.14159265358979323846);
  const double a = 0.044715;
  const double t = std::tanh(c * (z + a * z * z * z));
  return 0.5 * (1.0 + t) + 0.5 * z * (1.0 - t * t) * c * (1.0 + 3.0 * a * z * z);
}

bool valid_forward_epi(int epi) {
  return (epi >= ORA_NONE && epi <= ORA_RELU_AUX_BIAS) || epi == ORA_GELU_ERF_BIAS ||
         epi == ORA_GELU_AUX_BIAS;
}

template <class F>
void parallel_rows(int64_t rows, int nthreads, F fn) {
  if (nthreads <= 1 || rows < 2) {
    for (int64_t r = 0; r < rows; ++r) fn(r);
    return;
  }
  if (nthreads > rows) nthreads = (int)rows;
  std::vector<std::thread> pool;
  for (int t = 0; t < nthreads; ++t) {
    pool.emplace_back([=]() {
      for (int64_t r = t; r < rows; r += nthreads) fn(r);
    });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

double ora_f16_to_f64(uint16_t h) { return f16_decode(h); }
double ora_bf16_to_f64(uint16_t h) { return bf16_decode(h); }
uint16_t ora_f64_to_bf16(double x) { return bf16_encode(x); }
void ora_bf16_to_f64_array(const uint16_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_decode(in[i]);
}
void ora_f64_to_bf16_array(const double* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_encode(in[i]);
}
// The activation of epilogue `epi` applied to one fp64 pre-activation value
// (the same function the forward uses); -1 selects nothing and returns NaN.
double ora_act_f64(int epi, double z) {
  if (!valid_forward_epi(epi)) return std::nan("");
  return activation(epi, z);
}
uint16_t ora_f64_to_f16(double x) { return f16_encode(x); }

void ora_f16_to_f64_array(const uint16_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f16_decode(in[i]);
}
void ora_f64_to_f16_array(const double* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f16_encode(in[i]);
}

// D = act(A.B + bias) for the whole (M, N, K) problem.
//   A[m,k] at A[m*lda + k] when a_major == 0 (K-major), A[k*lda + m] when 1.
//   B[k,n] at B[n*ldb + k] when b_major == 0 (K-major), B[k*ldb + n] when 1.
//   D[m,n] at D[m*ldd + n] when d_layout == 0 (row),     D[n*ldd + m] when 1.
//   Stored row r / contiguous index c of D: (r,c) = (m,n) row, (n,m) col.
//   aux (RELU_AUX_BIAS only): bit (c % 32) of aux[r*ld_aux + c/32] = (z > 0);
//   every word of every stored row is written (padding bits 0).
//   Z (optional, may be NULL): the fp64 pre-activation z, laid out like D.
//   bias may be NULL only for ORA_NONE.
// Returns 0 on success, -1 on a bad argument.

}  // extern "C"

namespace {

// The forward with both kinds of auxiliary output: `aux` (bit mask, for
// RELU_AUX_BIAS) and `zaux` (the pre-activation rounded to the element type,
// for GELU_AUX_BIAS, at zaux[r*ld_zaux + c] in D's stored layout).
int forward_impl(int dt, int64_t M, int64_t N, int64_t K,
                 const uint16_t* A, int a_major, int64_t lda,
                 const uint16_t* B, int b_major, int64_t ldb,
                 const uint16_t* bias, int epi,
                 uint16_t* D, int d_layout, int64_t ldd,
                 uint32_t* aux, int64_t ld_aux, uint16_t* zaux, int64_t ld_zaux, double* Z,
                 int nthreads) {
  if (dt != 0 && dt != 1) return -1;
  if (M < 0 || N < 0 || K < 0 || !D) return -1;
  if (!valid_forward_epi(epi)) return -1;
  if (epi != ORA_NONE && !bias) return -1;
  if (epi == ORA_RELU_AUX_BIAS && !aux) return -1;
  if (epi == ORA_GELU_AUX_BIAS && !zaux) return -1;
  const int64_t rows = d_layout == 0 ? M : N;
  const int64_t cols = d_layout == 0 ? N : M;
  if (ldd < cols || (aux && ld_aux * 32 < cols) || (zaux && ld_zaux < cols)) return -1;
  if (K > 0 && (!A || !B)) return -1;

  // Layout step only: decode both operands into plain fp64 matrices with k
  // contiguous, Ad[m][k] = A[m,k] and Bd[n][k] = B[k,n]. The products of two
  // fp16 values are exact in fp64; the sums below run k = 0, 1, ..., K-1.
  std::vector<double> Ad((size_t)M * (size_t)K), Bd((size_t)N * (size_t)K);
  parallel_rows(M, nthreads, [&](int64_t m) {
    for (int64_t k = 0; k < K; ++k)
      Ad[m * K + k] = decode(dt, a_major == 0 ? A[m * lda + k] : A[k * lda + m]);
  });
  parallel_rows(N, nthreads, [&](int64_t n) {
    for (int64_t k = 0; k < K; ++k)
      Bd[n * K + k] = decode(dt, b_major == 0 ? B[n * ldb + k] : B[k * ldb + n]);
  });

  parallel_rows(rows, nthreads, [&](int64_t r) {
    if (epi == ORA_RELU_AUX_BIAS)
      std::memset(aux + r * ld_aux, 0, sizeof(uint32_t) * ld_aux);
    for (int64_t c = 0; c < cols; ++c) {
      const int64_t m = d_layout == 0 ? r : c;
      const int64_t n = d_layout == 0 ? c : r;
      const double* a = Ad.data() + m * K;
      const double* b = Bd.data() + n * K;
      double z = 0.0;
      for (int64_t k = 0; k < K; ++k) z += a[k] * b[k];
      if (epi != ORA_NONE) z += decode(dt, bias[m]);
      const double y = activation(epi, z);
      D[r * ldd + c] = encode(dt, y);
      if (Z) Z[r * ldd + c] = z;
      if (epi == ORA_RELU_AUX_BIAS && z > 0.0)
        aux[r * ld_aux + c / 32] |= (uint32_t)1u << (c % 32);
      if (epi == ORA_GELU_AUX_BIAS) zaux[r * ld_zaux + c] = encode(dt, z);
    }
  });
  return 0;
}

}  // namespace

extern "C" {

// Same as ora_linear_forward with every operand, the bias and D of element
// type `dt` (0 = fp16, 1 = bfloat16).
int ora_linear_forward_dt(int dt, int64_t M, int64_t N, int64_t K,
                          const uint16_t* A, int a_major, int64_t lda,
                          const uint16_t* B, int b_major, int64_t ldb,
                          const uint16_t* bias, int epi,
                          uint16_t* D, int d_layout, int64_t ldd,
                          uint32_t* aux, int64_t ld_aux, double* Z,
                          int nthreads) {
  if (epi == ORA_GELU_AUX_BIAS) return -1;  // needs the 16-bit z output below
  return forward_impl(dt, M, N, K, A, a_major, lda, B, b_major, ldb, bias, epi, D, d_layout, ldd,
                      aux, ld_aux, nullptr, 0, Z, nthreads);
}

// GELU_AUX_BIAS: D = tanh-GELU(z) as GELU_BIAS, and zaux = z rounded to the
// element type, stored like D (zaux[r*ld_zaux + c]); the backward pass
// (DGELU_BGRAD) reads it to evaluate the GELU derivative.
int ora_gelu_aux_forward_dt(int dt, int64_t M, int64_t N, int64_t K,
                            const uint16_t* A, int a_major, int64_t lda,
                            const uint16_t* B, int b_major, int64_t ldb,
                            const uint16_t* bias, uint16_t* D, int d_layout, int64_t ldd,
                            uint16_t* zaux, int64_t ld_zaux, double* Z, int nthreads) {
  return forward_impl(dt, M, N, K, A, a_major, lda, B, b_major, ldb, bias, ORA_GELU_AUX_BIAS, D,
                      d_layout, ldd, nullptr, 0, zaux, ld_zaux, Z, nthreads);
}

int ora_linear_forward(int64_t M, int64_t N, int64_t K,
                       const uint16_t* A, int a_major, int64_t lda,
                       const uint16_t* B, int b_major, int64_t ldb,
                       const uint16_t* bias, int epi,
                       uint16_t* D, int d_layout, int64_t ldd,
                       uint32_t* aux, int64_t ld_aux, double* Z,
                       int nthreads) {
  return ora_linear_forward_dt(0, M, N, K, A, a_major, lda, B, b_major, ldb, bias, epi, D,
                               d_layout, ldd, aux, ld_aux, Z, nthreads);
}

// DRELU_BGRAD as the epilogue of a GEMM (the backward product dH = A.B whose
// result is masked before it is stored), from the same description: the
// ReLU-gradient mask is applied to the product and the bias gradient is
// accumulated from the masked values.
//   z[m,n]    = sum_k A[m,k] B[k,n]           (fp64, k ascending; no bias)
//   dZ[m,n]   = fp16(z[m,n]) if bit(m,n) else +0
//   bgrad[m]  = sum over n of z[m,n]*bit(m,n)  (fp64, n ascending, unrounded z)
// Layouts as ora_linear_forward; aux is the forward mask in D's layout.
int ora_gemm_drelu_bgrad_dt(int dt, int64_t M, int64_t N, int64_t K,
                            const uint16_t* A, int a_major, int64_t lda,
                            const uint16_t* B, int b_major, int64_t ldb,
                            const uint32_t* aux, int64_t ld_aux,
                            uint16_t* dZ, int d_layout, int64_t ldd, double* bgrad,
                            int nthreads) {
  if (dt != 0 && dt != 1) return -1;
  if (M < 0 || N < 0 || K < 0 || !dZ || !aux || !bgrad) return -1;
  const int64_t cols = d_layout == 0 ? N : M;
  if (ldd < cols || ld_aux * 32 < cols) return -1;
  if (K > 0 && (!A || !B)) return -1;
  std::vector<double> Ad((size_t)M * (size_t)K), Bd((size_t)N * (size_t)K);
  parallel_rows(M, nthreads, [&](int64_t m) {
    for (int64_t k = 0; k < K; ++k)
      Ad[m * K + k] = decode(dt, a_major == 0 ? A[m * lda + k] : A[k * lda + m]);
  });
  parallel_rows(N, nthreads, [&](int64_t n) {
    for (int64_t k = 0; k < K; ++k)
      Bd[n * K + k] = decode(dt, b_major == 0 ? B[n * ldb + k] : B[k * ldb + n]);
  });
  parallel_rows(M, nthreads, [&](int64_t m) {
    double s = 0.0;
    for (int64_t n = 0; n < N; ++n) {
      const double* a = Ad.data() + m * K;
      const double* b = Bd.data() + n * K;
      double z = 0.0;
      for (int64_t k = 0; k < K; ++k) z += a[k] * b[k];
      const int64_t r = d_layout == 0 ? m : n;
      const int64_t c = d_layout == 0 ? n : m;
      const bool bit = (aux[r * ld_aux + c / 32] >> (c % 32)) & 1u;
      dZ[r * ldd + c] = bit ? encode(dt, z) : (uint16_t)0;
      if (bit) s += z;
    }
    bgrad[m] = s;
  });
  return 0;
}

int ora_gemm_drelu_bgrad(int64_t M, int64_t N, int64_t K,
                         const uint16_t* A, int a_major, int64_t lda,
                         const uint16_t* B, int b_major, int64_t ldb,
                         const uint32_t* aux, int64_t ld_aux,
                         uint16_t* dZ, int d_layout, int64_t ldd, double* bgrad,
                         int nthreads) {
  return ora_gemm_drelu_bgrad_dt(0, M, N, K, A, a_major, lda, B, b_major, ldb, aux, ld_aux, dZ,
                                 d_layout, ldd, bgrad, nthreads);
}

// Backward epilogue (DRELU_BGRAD), from the page's description: apply the
// stored ReLU mask to the incoming gradient and reduce the bias gradient.
//   dY, dZ: [M, N] in the forward D's stored layout (d_layout, ldd).
//   aux: the forward mask (same packing as ora_linear_forward).
//   dZ[m,n] = dY[m,n] if bit(m,n) else +0.
//   bgrad[m] = sum over n of dZ[m,n], n ascending, fp64.
int ora_drelu_bgrad_dt(int dt, int64_t M, int64_t N, const uint16_t* dY, int d_layout,
                       int64_t ldd, const uint32_t* aux, int64_t ld_aux,
                       uint16_t* dZ, double* bgrad) {
  if (dt != 0 && dt != 1) return -1;
  if (M < 0 || N < 0 || !dY || !aux || !dZ || !bgrad) return -1;
  for (int64_t m = 0; m < M; ++m) bgrad[m] = 0.0;
  for (int64_t m = 0; m < M; ++m) {
    double s = 0.0;
    for (int64_t n = 0; n < N; ++n) {
      const int64_t r = d_layout == 0 ? m : n;
      const int64_t c = d_layout == 0 ? n : m;
      const bool bit = (aux[r * ld_aux + c / 32] >> (c % 32)) & 1u;
      // ReLU'(z) is 1 where the mask bit is set and 0 elsewhere; a masked-out
      // gradient is +0 (a select, so -0, inf or NaN in dY do not leak).
      const uint16_t out = bit ? dY[r * ldd + c] : (uint16_t)0;
      dZ[r * ldd + c] = out;
      s += decode(dt, out);
    }
    bgrad[m] = s;
  }
  return 0;
}

int ora_drelu_bgrad(int64_t M, int64_t N, const uint16_t* dY, int d_layout,
                    int64_t ldd, const uint32_t* aux, int64_t ld_aux,
                    uint16_t* dZ, double* bgrad) {
  return ora_drelu_bgrad_dt(0, M, N, dY, d_layout, ldd, aux, ld_aux, dZ, bgrad);
}

}  // extern "C"

extern "C" {

// Derivative of the tanh-form GELU at one fp64 value (for the pins).
double ora_gelu_grad_f64(double z) { return gelu_tanh_grad(z); }

// DGELU_BGRAD standalone, the GELU counterpart of DRELU_BGRAD (cuBLASLt's
// backward epilogue family named on the nvmath-python bias-fusion guide,
// "Advanced techniques"): the incoming gradient is multiplied by the GELU
// derivative at the stored pre-activation, and the bias gradient is reduced.
//   dY, zaux, dZ: [M, N] in the forward D's stored layout (d_layout, ldd);
//   zaux holds z rounded to the element type (GELU_AUX_BIAS's output).
//   g[m,n]    = dY[m,n] * gelu'(z[m,n])          (fp64)
//   dZ[m,n]   = g[m,n] rounded to the element type
//   bgrad[m]  = sum over n of g[m,n]              (fp64, unrounded g)
int ora_dgelu_bgrad_dt(int dt, int64_t M, int64_t N, const uint16_t* dY, int d_layout,
                       int64_t ldd, const uint16_t* zaux, int64_t ld_zaux,
                       uint16_t* dZ, double* bgrad) {
  if (dt != 0 && dt != 1) return -1;
  if (M < 0 || N < 0 || !dY || !zaux || !dZ || !bgrad) return -1;
  const int64_t cols = d_layout == 0 ? N : M;
  if (ldd < cols || ld_zaux < cols) return -1;
  for (int64_t m = 0; m < M; ++m) {
    double s = 0.0;
    for (int64_t n = 0; n < N; ++n) {
      const int64_t r = d_layout == 0 ? m : n;
      const int64_t c = d_layout == 0 ? n : m;
      const double g = decode(dt, dY[r * ldd + c]) * gelu_tanh_grad(decode(dt, zaux[r * ld_zaux + c]));
      dZ[r * ldd + c] = encode(dt, g);
      s += g;
    }
    bgrad[m] = s;
  }
  return 0;
}

// DGELU_BGRAD as the epilogue of the backward GEMM: the product dH = A.B
// (fp64, k ascending) takes the place of dY above.
//   dZ[m,n]  = (dH[m,n] * gelu'(z[m,n])) rounded to the element type
//   bgrad[m] = sum over n of dH[m,n] * gelu'(z[m,n])   (fp64, n ascending)
int ora_gemm_dgelu_bgrad_dt(int dt, int64_t M, int64_t N, int64_t K,
                            const uint16_t* A, int a_major, int64_t lda,
                            const uint16_t* B, int b_major, int64_t ldb,
                            const uint16_t* zaux, int64_t ld_zaux,
                            uint16_t* dZ, int d_layout, int64_t ldd, double* bgrad,
                            int nthreads) {
  if (dt != 0 && dt != 1) return -1;
  if (M < 0 || N < 0 || K < 0 || !dZ || !zaux || !bgrad) return -1;
  const int64_t cols = d_layout == 0 ? N : M;
  if (ldd < cols || ld_zaux < cols) return -1;
  if (K > 0 && (!A || !B)) return -1;
  std::vector<double> Ad((size_t)M * (size_t)K), Bd((size_t)N * (size_t)K);
  parallel_rows(M, nthreads, [&](int64_t m) {
    for (int64_t k = 0; k < K; ++k)
      Ad[m * K + k] = decode(dt, a_major == 0 ? A[m * lda + k] : A[k * lda + m]);
  });
  parallel_rows(N, nthreads, [&](int64_t n) {
    for (int64_t k = 0; k < K; ++k)
      Bd[n * K + k] = decode(dt, b_major == 0 ? B[n * ldb + k] : B[k * ldb + n]);
  });
  parallel_rows(M, nthreads, [&](int64_t m) {
    double s = 0.0;
    for (int64_t n = 0; n < N; ++n) {
      const double* a = Ad.data() + m * K;
      const double* b = Bd.data() + n * K;
      double h = 0.0;
      for (int64_t k = 0; k < K; ++k) h += a[k] * b[k];
      const int64_t r = d_layout == 0 ? m : n;
      const int64_t c = d_layout == 0 ? n : m;
      const double g = h * gelu_tanh_grad(decode(dt, zaux[r * ld_zaux + c]));
      dZ[r * ldd + c] = encode(dt, g);
      s += g;
    }
    bgrad[m] = s;
  });
  return 0;
}

}  // extern "C"

extern "C" {

// MatMul + bias + residual + normalisation over the output features: the
// structural fusion of ops-nn MatMul fusion (codearts), "ops-nn's MatMul
// fusion strategy", second level (MatMul + LayerNorm / RMSNorm + residual,
// where the norm reduces across the channel dimension).
//   h[m,n] = sum_k A[m,k] B[k,n] + bias[m] + res[m,n]      (fp64)
//   H[m,n] = h rounded to the element type (the new residual stream)
// for every token n, over the M features m (population statistics):
//   kind 0, RMSNorm:   y = h / sqrt(mean_m(h^2) + eps) * gamma[m]
//   kind 1, LayerNorm: y = (h - mu) / sqrt(mean_m((h - mu)^2) + eps) * gamma[m]
//                          + beta[m],   mu = mean_m(h)
//   Y[m,n] = y rounded to the element type.
// res, H and Y are stored like D (d_layout, ldd); gamma and beta are [M]
// vectors of the element type (beta unused by RMSNorm). Statistics use the
// unrounded fp64 h, summed in ascending m.
int ora_linear_norm_dt(int dt, int kind, int64_t M, int64_t N, int64_t K,
                       const uint16_t* A, int a_major, int64_t lda,
                       const uint16_t* B, int b_major, int64_t ldb,
                       const uint16_t* bias, const uint16_t* res,
                       const uint16_t* gamma, const uint16_t* beta, double eps,
                       uint16_t* H, uint16_t* Y, int d_layout, int64_t ldd, int nthreads) {
  if (dt != 0 && dt != 1) return -1;
  if (kind != 0 && kind != 1) return -1;
  if (M < 1 || N < 0 || K < 0 || !bias || !res || !gamma || !H || !Y) return -1;
  if (kind == 1 && !beta) return -1;
  if (!(eps >= 0.0)) return -1;
  const int64_t cols = d_layout == 0 ? N : M;
  if (ldd < cols) return -1;
  if (K > 0 && (!A || !B)) return -1;
  std::vector<double> Ad((size_t)M * (size_t)K), Bd((size_t)N * (size_t)K);
  parallel_rows(M, nthreads, [&](int64_t m) {
    for (int64_t k = 0; k < K; ++k)
      Ad[m * K + k] = decode(dt, a_major == 0 ? A[m * lda + k] : A[k * lda + m]);
  });
  parallel_rows(N, nthreads, [&](int64_t n) {
    for (int64_t k = 0; k < K; ++k)
      Bd[n * K + k] = decode(dt, b_major == 0 ? B[n * ldb + k] : B[k * ldb + n]);
  });
  auto at = [&](int64_t m, int64_t n) { return d_layout == 0 ? m * ldd + n : n * ldd + m; };
  parallel_rows(N, nthreads, [&](int64_t n) {
    std::vector<double> h((size_t)M);
    for (int64_t m = 0; m < M; ++m) {
      const double* a = Ad.data() + m * K;
      const double* b = Bd.data() + n * K;
      double z = 0.0;
      for (int64_t k = 0; k < K; ++k) z += a[k] * b[k];
      h[m] = z + decode(dt, bias[m]) + decode(dt, res[at(m, n)]);
      H[at(m, n)] = encode(dt, h[m]);
    }
    double mu = 0.0;
    if (kind == 1) {
      for (int64_t m = 0; m < M; ++m) mu += h[m];
      mu /= (double)M;
    }
    double ss = 0.0;
    for (int64_t m = 0; m < M; ++m) ss += (h[m] - mu) * (h[m] - mu);
    const double inv = 1.0 / std::sqrt(ss / (double)M + eps);
    for (int64_t m = 0; m < M; ++m) {
      double y = (h[m] - mu) * inv * decode(dt, gamma[m]);
      if (kind == 1) y += decode(dt, beta[m]);
      Y[at(m, n)] = encode(dt, y);
    }
  });
  return 0;
}

}  // extern "C"
