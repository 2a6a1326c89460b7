// ge_unfused.cu -- the unfused baseline's elementwise kernels, and the
// bounded-wait probe used by the failure-path test.
//
// ops-nn MatMul fusion (codearts), "ops-nn's MatMul fusion strategy", first
// level: without fusion the product is written to HBM, read back for the
// bias add and written again, then read back for the activation and written
// again. These two kernels are those extra passes; with the GEMM's NONE
// epilogue in front they form the three-kernel baseline the fused path is
// measured against. Both work in place on D and are bound by HBM bandwidth.
#include "ge_internal.h"
#include "ge_ptx.cuh"

namespace ge {
namespace {

__device__ __forceinline__ float act_of(int epi, float z) {
  if (epi == EPI_RELU_BIAS || epi == EPI_RELU_AUX_BIAS) return fmaxf(z, 0.0f);
  if (epi == EPI_GELU_BIAS || epi == EPI_GELU_AUX_BIAS) return gelu_tanh(z);
  if (epi == EPI_GELU_ERF_BIAS) return gelu_erf(z);
  return z;
}

// D[r, c] += bias[r] (bias_per_row) or bias[c]; 8 contiguous fp16 per thread.
__global__ void __launch_bounds__(256) bias_add_kernel(__half* D, long long R, long long C,
                                                        long long ld, const __half* bias,
                                                        int bias_per_row, int bf16_flag) {
  const bool bf16 = bf16_flag != 0;
  const unsigned short* b16 = reinterpret_cast<const unsigned short*>(bias);
  const long long vpr = (C + 7) / 8;  // 8-wide groups per row
  const long long total = R * vpr;
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < total; i += gridDim.x * 256LL) {
    const long long r = i / vpr;
    const long long c0 = (i - r * vpr) * 8;
    unsigned short* row = reinterpret_cast<unsigned short*>(D) + r * ld;
    if (c0 + 8 <= C) {
      uint4 v = *reinterpret_cast<const uint4*>(row + c0);
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        float2 f = to_f32x2(bf16, w[t]);
        f.x += to_f32(bf16, bias_per_row ? b16[r] : b16[c0 + 2 * t]);
        f.y += to_f32(bf16, bias_per_row ? b16[r] : b16[c0 + 2 * t + 1]);
        w[t] = pack2(bf16, f.x, f.y);
      }
      *reinterpret_cast<uint4*>(row + c0) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      for (long long c = c0; c < C; ++c)
        row[c] = from_f32(bf16, to_f32(bf16, row[c]) + to_f32(bf16, bias_per_row ? b16[r] : b16[c]));
    }
  }
}

// D = act(D) in place, 8 contiguous fp16 per lane (a warp reads 512
// contiguous bytes). With a mask, four consecutive lanes cover one 32-element
// mask word: each builds its byte and lane 0 of the four writes the word
// (padding words up to the row's 128-column boundary included).
__global__ void __launch_bounds__(256) activation_kernel(__half* D, long long R, long long C,
                                                          long long ld, int epi, uint32_t* aux,
                                                          long long ld_aux, unsigned short* zaux,
                                                          long long ld_zaux, int bf16_flag) {
  const bool bf16 = bf16_flag != 0;
  const long long wpr = aux ? ld_aux : (C + 31) / 32;  // 32-element words per row
  const long long units = R * wpr * 4;                 // one unit = 8 elements
  const long long pad_cols = ((C + 127) / 128) * 128;
  // the loop bound is a multiple of 32 so whole warps iterate together
  const long long total = (units + 31) & ~31LL;
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < total; i += gridDim.x * 256LL) {
    uint32_t byte = 0;
    long long r = 0, word = 0, c0 = 0;
    const bool live = i < units;
    if (live) {
      const long long u = i >> 2;
      r = u / wpr;
      word = u - r * wpr;
      c0 = word * 32 + (i & 3) * 8;
      unsigned short* row = reinterpret_cast<unsigned short*>(D) + r * ld;
      if (c0 + 8 <= C) {
        uint4 v = *reinterpret_cast<const uint4*>(row + c0);
        if (zaux) *reinterpret_cast<uint4*>(zaux + r * ld_zaux + c0) = v;  // GELU_AUX_BIAS: keep z
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float2 f = to_f32x2(bf16, w[t]);
          byte |= (f.x > 0.0f ? 1u : 0u) << (2 * t);
          byte |= (f.y > 0.0f ? 1u : 0u) << (2 * t + 1);
          w[t] = pack2(bf16, act_of(epi, f.x), act_of(epi, f.y));
        }
        *reinterpret_cast<uint4*>(row + c0) = make_uint4(w[0], w[1], w[2], w[3]);
      } else {
        for (long long c = c0; c < C && c < c0 + 8; ++c) {
          if (zaux) zaux[r * ld_zaux + c] = row[c];
          const float f = to_f32(bf16, row[c]);
          byte |= (f > 0.0f ? 1u : 0u) << (c - c0);
          row[c] = from_f32(bf16, act_of(epi, f));
        }
      }
    }
    if (aux && epi == EPI_RELU_AUX_BIAS) {
      const int lane = threadIdx.x & 31;
      const int base = lane & ~3;
      uint32_t wv = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) wv |= __shfl_sync(0xffffffffu, byte, base + q) << (8 * q);
      if (live && (lane & 3) == 0 && word * 32 < pad_cols) aux[r * ld_aux + word] = wv;
    }
  }
}

__global__ void wait_probe_kernel(unsigned int* err, long long budget) {
  __shared__ __align__(8) unsigned long long bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nobody ever arrives on `bar`: the wait must give up after `budget`.
    if (!mbar_wait_bounded(smem_u32(&bar), 0u, &abort_flag, budget)) atomicOr(err, ERR_PROBE_TIMEOUT);
  }
}

int grid_for(long long work, int per_block) {
  long long b = (work + per_block - 1) / per_block;
  if (b > 65535LL * 8) b = 65535LL * 8;
  if (b < 1) b = 1;
  return static_cast<int>(b);
}

}  // namespace

cudaError_t launch_bias_add(__half* D, long long R, long long C, long long ld, const __half* bias,
                            int bias_per_row, int bf16, cudaStream_t s) {
  if (R == 0 || C == 0) return cudaSuccess;
  bias_add_kernel<<<grid_for(R * ((C + 7) / 8), 256), 256, 0, s>>>(D, R, C, ld, bias, bias_per_row, bf16);
  return cudaGetLastError();
}

cudaError_t launch_activation(__half* D, long long R, long long C, long long ld, int epi,
                              uint32_t* aux, long long ld_aux, unsigned short* zaux,
                              long long ld_zaux, int bf16, cudaStream_t s) {
  if (R == 0 || C == 0) return cudaSuccess;
  const long long wpr = aux ? ld_aux : (C + 31) / 32;
  activation_kernel<<<grid_for(R * wpr * 4, 256), 256, 0, s>>>(D, R, C, ld, epi, aux, ld_aux, zaux,
                                                               ld_zaux, bf16);
  return cudaGetLastError();
}

cudaError_t launch_wait_probe(unsigned int* err, long long budget, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(err, budget);
  return cudaGetLastError();
}

}  // namespace ge
