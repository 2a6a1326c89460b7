// ge_gemv.cu -- weight-streaming GEMV with the fused bias + activation
// epilogue, for token counts N <= 16 (decode).
//
// ops-nn MatMul fusion (codearts), "Why MatMul is the inference bottleneck":
// with one token per step the activation is [1, hidden] against a
// [hidden, hidden] weight, the product has almost no reuse, and its time is
// the time to read the weight once from HBM; the fused epilogue then costs
// nothing extra because the result never leaves the chip before the bias and
// activation are applied ("ops-nn's MatMul fusion strategy", first level).
//
// One warp owns one weight row at a time and streams it with 16-byte
// non-allocating loads (8 fp16 per lane, UNROLL slabs in flight); the N
// activation vectors are small and stay in L1/L2. fp32 accumulation, a
// butterfly warp reduction, then bias + activation + fp16 rounding per output.
#include "ge_internal.h"
#include "ge_ptx.cuh"

namespace ge {
namespace {

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float dot8(const uint4& a, const uint4& b, float acc) {
  const __half2* ha = reinterpret_cast<const __half2*>(&a);
  const __half2* hb = reinterpret_cast<const __half2*>(&b);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fa = __half22float2(ha[i]);
    const float2 fb = __half22float2(hb[i]);
    acc = fmaf(fa.x, fb.x, acc);
    acc = fmaf(fa.y, fb.y, acc);
  }
  return acc;
}

template <int NT, int UNROLL>
__global__ void __launch_bounds__(256) gemv_kernel(const GemvArgs p) {
  const int lane = threadIdx.x & 31;
  const long long wpb = blockDim.x >> 5;
  const long long nwarps = static_cast<long long>(gridDim.x) * wpb;
  const int K8 = p.K & ~7;
  constexpr int SLAB = 32 * 8;  // elements one warp covers per 16-byte load
  for (long long m = blockIdx.x * wpb + (threadIdx.x >> 5); m < p.M; m += nwarps) {
    const __half* arow = p.A + m * p.lda;
    float acc[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n] = 0.0f;
    int k = lane * 8;
    for (; k + (UNROLL - 1) * SLAB < K8; k += UNROLL * SLAB) {
      uint4 a[UNROLL];
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) a[u] = ld_stream(arow + k + u * SLAB);
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        if (n < p.N) {
          const __half* brow = p.B + n * p.ldb + k;
#pragma unroll
          for (int u = 0; u < UNROLL; ++u)
            acc[n] = dot8(a[u], __ldg(reinterpret_cast<const uint4*>(brow + u * SLAB)), acc[n]);
        }
      }
    }
    for (; k < K8; k += SLAB) {
      const uint4 a = ld_stream(arow + k);
#pragma unroll
      for (int n = 0; n < NT; ++n)
        if (n < p.N) acc[n] = dot8(a, __ldg(reinterpret_cast<const uint4*>(p.B + n * p.ldb + k)), acc[n]);
    }
    for (int kk = K8 + lane; kk < p.K; kk += 32) {  // ragged K tail
      const float av = __half2float(arow[kk]);
#pragma unroll
      for (int n = 0; n < NT; ++n)
        if (n < p.N) acc[n] = fmaf(av, __half2float(p.B[n * p.ldb + kk]), acc[n]);
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[n] += __shfl_xor_sync(0xffffffffu, acc[n], off);
    }
    float z = 0.0f;
#pragma unroll
    for (int n = 0; n < NT; ++n)
      if (n == lane) z = acc[n];
    if (lane < p.N) {
      if (p.epi != EPI_NONE) z += __half2float(p.bias[m]);
      float y = z;
      if (p.epi == EPI_RELU_BIAS) y = fmaxf(z, 0.0f);
      else if (p.epi == EPI_GELU_BIAS) y = gelu_tanh(z);
      p.D[m * p.ldd_m + static_cast<long long>(lane) * p.ldd_n] = __float2half_rn(y);
    }
  }
}

template <int NT, int UNROLL>
cudaError_t launch_nt(const GemvArgs& a, int num_sms, cudaStream_t s) {
  constexpr int threads = 256;
  long long blocks = (a.M + 7) / 8;  // one row per warp when the grid allows
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  gemv_kernel<NT, UNROLL><<<static_cast<int>(blocks), threads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const GemvArgs& a, int num_sms, cudaStream_t s) {
  if (a.N <= 1) return launch_nt<1, 8>(a, num_sms, s);
  if (a.N <= 2) return launch_nt<2, 8>(a, num_sms, s);
  if (a.N <= 4) return launch_nt<4, 4>(a, num_sms, s);
  if (a.N <= 8) return launch_nt<8, 4>(a, num_sms, s);
  return launch_nt<16, 2>(a, num_sms, s);
}

}  // namespace ge
