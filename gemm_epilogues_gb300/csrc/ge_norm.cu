// ge_norm.cu -- the normalisation pass of MatMul + bias + residual +
// RMSNorm / LayerNorm (ops-nn MatMul fusion (codearts), "ops-nn's MatMul
// fusion strategy", second level: the norm reduces across the channel
// dimension, so it cannot be applied element by element in the GEMM's
// epilogue). The GEMM epilogue has already written h = A.B + bias +
// residual as H; this kernel reads every token's row of H once and writes
// the normalised row:
//
//   RMSNorm:   y = h * rsqrt(mean(h^2) + eps) * gamma
//   LayerNorm: y = (h - mu) * rsqrt(mean((h - mu)^2) + eps) * gamma + beta
//
// One warp per row. The row stays in registers (up to CACHE 16-byte groups
// per lane, 4096 16-bit features), so the mean and the variance are two
// exact passes over registers rather than a sum of squares minus a squared
// mean; longer rows re-read their remainder (from L2) in each pass. Memory
// traffic is one read of H and one write of Y: HBM-bound.
#include "ge_internal.h"
#include "ge_ptx.cuh"

namespace ge {
namespace {

constexpr int CACHE = 16;  // 16-byte groups per lane kept in registers

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(void* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return s;
}

// Sum over the eight 16-bit values of `v` of f(x).
template <class F>
__device__ __forceinline__ float sum8(const uint4& v, bool bf16, F f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = to_f32x2(bf16, w[i]);
    s += f(x.x) + f(x.y);
  }
  return s;
}

__global__ void __launch_bounds__(256) norm_kernel(const NormArgs p) {
  const bool bf16 = p.bf16 != 0;
  const int lane = threadIdx.x & 31;
  const long long wpb = blockDim.x >> 5;
  const long long nwarps = static_cast<long long>(gridDim.x) * wpb;
  const long long G = p.C >> 3;  // whole 16-byte groups per row
  const float inv_c = 1.0f / static_cast<float>(p.C);
  for (long long r = blockIdx.x * wpb + (threadIdx.x >> 5); r < p.R; r += nwarps) {
    const unsigned short* h = p.H + r * p.ld;
    unsigned short* y = p.Y + r * p.ld;
    uint4 cache[CACHE];
#pragma unroll
    for (int i = 0; i < CACHE; ++i) {
      const long long g = lane + 32LL * i;
      cache[i] = g < G ? ld_stream(h + 8 * g) : make_uint4(0, 0, 0, 0);
    }
    // Visit every 16-byte group g of the row owned by this lane: the cached
    // ones with static register indices, the rest (rows longer than
    // 32 * CACHE groups) re-read.
    auto for_groups = [&](auto&& fn) {
#pragma unroll
      for (int i = 0; i < CACHE; ++i) {
        const long long g = lane + 32LL * i;
        if (g < G) fn(cache[i], g);
      }
      for (long long g = lane + 32LL * CACHE; g < G; g += 32) fn(ld_stream(h + 8 * g), g);
    };
    // ragged tail (C % 8 elements): one element per lane
    const long long tail_c = 8 * G + lane;
    const bool has_tail = tail_c < p.C;
    const float tail = has_tail ? to_f32(bf16, h[tail_c]) : 0.0f;

    float mu = 0.0f;
    if (p.layer) {
      float s = tail;
      for_groups([&](const uint4& v, long long) { s += sum8(v, bf16, [](float x) { return x; }); });
      mu = warp_sum(s) * inv_c;
    }
    float ss = has_tail ? (tail - mu) * (tail - mu) : 0.0f;
    for_groups([&](const uint4& v, long long) {
      ss += sum8(v, bf16, [mu](float x) { return (x - mu) * (x - mu); });
    });
    const float rstd = rsqrtf(warp_sum(ss) * inv_c + p.eps);

    for_groups([&](const uint4& v, long long g) {
      const uint4 gm = __ldg(reinterpret_cast<const uint4*>(p.gamma + 8 * g));
      uint4 bt = make_uint4(0, 0, 0, 0);
      if (p.layer) bt = __ldg(reinterpret_cast<const uint4*>(p.beta + 8 * g));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      const uint32_t gw[4] = {gm.x, gm.y, gm.z, gm.w};
      const uint32_t bw[4] = {bt.x, bt.y, bt.z, bt.w};
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 x = to_f32x2(bf16, w[k]);
        const float2 gg = to_f32x2(bf16, gw[k]);
        const float2 bb = p.layer ? to_f32x2(bf16, bw[k]) : make_float2(0.0f, 0.0f);
        o[k] = pack2(bf16, fmaf((x.x - mu) * rstd, gg.x, bb.x), fmaf((x.y - mu) * rstd, gg.y, bb.y));
      }
      st_stream(y + 8 * g, make_uint4(o[0], o[1], o[2], o[3]));
    });
    if (has_tail) {
      const float gg = to_f32(bf16, p.gamma[tail_c]);
      const float bb = p.layer ? to_f32(bf16, p.beta[tail_c]) : 0.0f;
      y[tail_c] = from_f32(bf16, fmaf((tail - mu) * rstd, gg, bb));
    }
  }
}

__global__ void __launch_bounds__(256) residual_add_kernel(unsigned short* D, long long R, long long C,
                                                           long long ld, const unsigned short* res,
                                                           int bf16_flag) {
  const bool bf16 = bf16_flag != 0;
  const long long per_row = (C + 7) / 8;
  const long long total = R * per_row;
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < total; i += gridDim.x * 256LL) {
    const long long r = i / per_row;
    const long long c0 = (i - r * per_row) * 8;
    unsigned short* d = D + r * ld + c0;
    const unsigned short* s = res + r * ld + c0;
    if (c0 + 8 <= C) {
      const uint4 a = *reinterpret_cast<const uint4*>(d);
      const uint4 b = *reinterpret_cast<const uint4*>(s);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
      const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 x = to_f32x2(bf16, aw[k]);
        const float2 z = to_f32x2(bf16, bw[k]);
        o[k] = pack2(bf16, x.x + z.x, x.y + z.y);
      }
      *reinterpret_cast<uint4*>(d) = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
      for (long long c = 0; c < C - c0; ++c) d[c] = from_f32(bf16, to_f32(bf16, d[c]) + to_f32(bf16, s[c]));
    }
  }
}

}  // namespace

cudaError_t launch_norm(const NormArgs& a, int num_sms, cudaStream_t s) {
  if (a.R == 0 || a.C == 0) return cudaSuccess;
  long long blocks = (a.R + 7) / 8;  // one row per warp when the grid allows
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  norm_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_residual_add(__half* D, long long R, long long C, long long ld,
                                const unsigned short* res, int bf16, cudaStream_t s) {
  if (R == 0 || C == 0) return cudaSuccess;
  long long blocks = (R * ((C + 7) / 8) + 255) / 256;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  residual_add_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(reinterpret_cast<unsigned short*>(D), R, C, ld,
                                                                    res, bf16);
  return cudaGetLastError();
}

}  // namespace ge
