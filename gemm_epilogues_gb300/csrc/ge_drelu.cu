// ge_drelu.cu -- DRELU_BGRAD: apply the stored ReLU mask to the incoming
// gradient and reduce the bias gradient, in one pass over dY.
//
// nvmath-python cuBLASLt bias-fusion guide, "Advanced techniques" (backward
// item): in training, the forward's fused ReLU needs a fused backward that
// applies the ReLU gradient mask and accumulates the bias gradient together.
// Fusing bias addition with matrix multiplication using nvmath-python: the
// mask is the auxiliary output RELU_AUX_BIAS keeps for this step.
//
//   dZ[m,n]  = dY[m,n] if mask(m,n) else +0
//   bgrad[m] = sum over n of dZ[m,n]        (fp32, fixed order)
//
// The work is a stream over dY (read once, 16-byte loads), the mask (1/16 of
// dY) and dZ (written once): bound by HBM bandwidth.
//
// Column case (D column-major: rows of storage are tokens n, the contiguous
// index is m, so bgrad is a sum down each storage column): a block covers
// 256 contiguous columns (32 lanes x 8 fp16) and one of `splits` row ranges;
// its 8 warps interleave rows; the warps' partial sums are combined in shared
// memory in a fixed order, written to a [splits][C] partial buffer, and the
// last block of a column strip (an atomic ticket) adds the splits in order.
// Row case (D row-major: bgrad is a sum along each storage row): one warp per
// row, 16-byte loads along the row, a butterfly reduction.
#include <cstdlib>

#include "ge_internal.h"
#include "ge_ptx.cuh"

namespace ge {
namespace {

constexpr int COLS_PER_BLOCK = 256;
constexpr int ROW_PHASES = 8;  // warps per block in the column case
constexpr int UNROLL = 8;      // rows in flight per thread (8 x 16 B loads)
constexpr int MIN_BLOCKS = 3;  // resident blocks per SM the register budget allows

// dZ may alias dY, so dY is read through the coherent path (no .nc).
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

// Keep the fp16 lanes of `v` whose mask bit (bits 0..7 of `bits`) is set,
// zero the others, and add the kept values to acc[0..7].
__device__ __forceinline__ uint4 mask_accumulate(uint4 v, uint32_t bits, float (&acc)[8]) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t keep = ((bits >> (2 * i)) & 1u ? 0x0000FFFFu : 0u) |
                          ((bits >> (2 * i + 1)) & 1u ? 0xFFFF0000u : 0u);
    w[i] &= keep;
    const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
    const float2 f = __half22float2(h);
    acc[2 * i] += f.x;
    acc[2 * i + 1] += f.y;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void __launch_bounds__(256, MIN_BLOCKS) drelu_cols_kernel(const DreluArgs p) {
  const int tx = threadIdx.x & 31;
  const int ty = threadIdx.x >> 5;
  const long long c0 = static_cast<long long>(blockIdx.x) * COLS_PER_BLOCK + tx * 8;
  const long long rows_per = (p.R + p.splits - 1) / p.splits;
  const long long r_begin = static_cast<long long>(blockIdx.y) * rows_per;
  const long long r_end = min(p.R, r_begin + rows_per);
  const bool full = c0 + 8 <= p.C;
  const int bit_off = static_cast<int>(c0 & 31);
  const long long widx = c0 >> 5;
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.0f;

  if (c0 < p.C) {
    long long r = r_begin + ty;
    if (full) {
      for (; r + (UNROLL - 1) * ROW_PHASES < r_end; r += UNROLL * ROW_PHASES) {
        uint4 v[UNROLL];
        uint32_t w[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
          const long long rr = r + u * ROW_PHASES;
          v[u] = ld_stream(p.dY + rr * p.ld + c0);
          w[u] = __ldg(p.mask + rr * p.ld_aux + widx);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
          const long long rr = r + u * ROW_PHASES;
          const uint4 o = mask_accumulate(v[u], w[u] >> bit_off, acc);
          st_stream(p.dZ + rr * p.ld + c0, o);
        }
      }
      for (; r < r_end; r += ROW_PHASES) {
        const uint4 v = ld_stream(p.dY + r * p.ld + c0);
        const uint32_t w = __ldg(p.mask + r * p.ld_aux + widx);
        st_stream(p.dZ + r * p.ld + c0, mask_accumulate(v, w >> bit_off, acc));
      }
    } else {
      for (; r < r_end; r += ROW_PHASES) {  // ragged last strip: element-wise
        const uint32_t w = __ldg(p.mask + r * p.ld_aux + widx) >> bit_off;
        for (int j = 0; j < 8 && c0 + j < p.C; ++j) {
          const __half g = p.dY[r * p.ld + c0 + j];
          const __half o = (w >> j) & 1u ? g : __ushort_as_half(0);
          p.dZ[r * p.ld + c0 + j] = o;
          acc[j] += __half2float(o);
        }
      }
    }
  }

  __shared__ float red[ROW_PHASES][COLS_PER_BLOCK];
  __shared__ unsigned int ticket;
#pragma unroll
  for (int j = 0; j < 8; ++j) red[ty][tx * 8 + j] = acc[j];
  __syncthreads();
  const long long c = static_cast<long long>(blockIdx.x) * COLS_PER_BLOCK + threadIdx.x;
  float s = 0.0f;
#pragma unroll
  for (int y = 0; y < ROW_PHASES; ++y) s += red[y][threadIdx.x];
  if (p.splits == 1) {
    if (c < p.C) p.bgrad[c] = s;
    return;
  }
  if (c < p.C) p.partials[static_cast<long long>(blockIdx.y) * p.C + c] = s;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) ticket = atomicAdd(p.counters + blockIdx.x, 1u);
  __syncthreads();
  if (ticket == static_cast<unsigned int>(p.splits - 1)) {
    // Last block of this strip: every split's partial is visible; add them
    // in split order so the result does not depend on block timing.
    __threadfence();
    if (c < p.C) {
      float t = 0.0f;
      for (int sp = 0; sp < p.splits; ++sp) t += __ldcg(p.partials + static_cast<long long>(sp) * p.C + c);
      p.bgrad[c] = t;
    }
    if (threadIdx.x == 0) p.counters[blockIdx.x] = 0u;  // ready for the next launch
  }
}

__global__ void __launch_bounds__(256) drelu_rows_kernel(const DreluArgs p) {
  const int lane = threadIdx.x & 31;
  const long long wpb = blockDim.x >> 5;
  const long long nwarps = static_cast<long long>(gridDim.x) * wpb;
  const long long C8 = p.C & ~7LL;
  for (long long r = blockIdx.x * wpb + (threadIdx.x >> 5); r < p.R; r += nwarps) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    const __half* src = p.dY + r * p.ld;
    __half* dst = p.dZ + r * p.ld;
    const uint32_t* mrow = p.mask + r * p.ld_aux;
    for (long long c = lane * 8; c < C8; c += 256) {
      const uint4 v = ld_stream(src + c);
      const uint32_t w = __ldg(mrow + (c >> 5)) >> (c & 31);
      st_stream(dst + c, mask_accumulate(v, w, acc));
    }
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += acc[j];
    for (long long c = C8 + lane; c < p.C; c += 32) {  // ragged tail
      const uint32_t w = (__ldg(mrow + (c >> 5)) >> (c & 31)) & 1u;
      const __half o = w ? src[c] : __ushort_as_half(0);
      dst[c] = o;
      s += __half2float(o);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) p.bgrad[r] = s;
  }
}

}  // namespace

// Row splits for the column case: about 1.3 waves of resident blocks (the
// fastest setting measured for dY[8192, 11008] with 3 blocks per SM: 14
// splits, 68 us against 72 us for two waves), at least 64 rows per split, at
// most 256 splits. GE_DRELU_SPLITS overrides (sweeps).
int drelu_splits(long long R, long long C, int num_sms) {
  static int occ = 0;
  if (occ == 0) {
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, drelu_cols_kernel, 256, 0) != cudaSuccess || o < 1) {
      cudaGetLastError();
      o = MIN_BLOCKS;
    }
    occ = o;
  }
  const long long strips = (C + COLS_PER_BLOCK - 1) / COLS_PER_BLOCK;
  long long want = (4LL * occ * num_sms / 3 + strips - 1) / strips;
  if (const char* env = std::getenv("GE_DRELU_SPLITS")) {
    const long long v = std::atoll(env);
    if (v >= 1) want = v;
  }
  const long long max_by_rows = (R + 63) / 64;
  if (want > max_by_rows) want = max_by_rows;
  if (want > 256) want = 256;
  if (want < 1) want = 1;
  return static_cast<int>(want);
}

cudaError_t launch_drelu_bgrad(const DreluArgs& a, int reduce_rows, cudaStream_t s) {
  if (a.R == 0 || a.C == 0) return cudaSuccess;
  if (reduce_rows) {
    const long long strips = (a.C + COLS_PER_BLOCK - 1) / COLS_PER_BLOCK;
    dim3 grid(static_cast<unsigned>(strips), static_cast<unsigned>(a.splits));
    drelu_cols_kernel<<<grid, 256, 0, s>>>(a);
  } else {
    long long blocks = (a.R + 7) / 8;
    if (blocks > 65535LL * 16) blocks = 65535LL * 16;
    drelu_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace ge
