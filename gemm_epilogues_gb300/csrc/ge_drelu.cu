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
// DGELU_BGRAD, the same pass for a GELU_AUX_BIAS forward, reads the stored
// pre-activation z (16-bit, laid out like dY) instead of mask bits:
//   dZ[m,n]  = dY[m,n] * gelu'(z[m,n])      (fp32 product, rounded once)
//   bgrad[m] = sum over n of the fp32 products
// (the GELU counterpart of the backward epilogue on the same pages).
//
// Column case (D column-major: rows of storage are tokens n, the contiguous
// index is m, so bgrad is a sum down each storage column): a block covers
// 256 contiguous columns (32 lanes x 8 fp16) and one of `splits` row ranges;
// its 8 warps interleave rows; the warps' partial sums are combined in shared
// memory in a fixed order, written to a [splits][C] partial buffer, and the
// last block of a column strip (an atomic ticket) adds the splits in order.
// Row case (D row-major: bgrad is a sum along each storage row): one warp per
// row, 16-byte loads along the row, a butterfly reduction.
#include <atomic>
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
__device__ __forceinline__ uint4 mask_accumulate(uint4 v, uint32_t bits, float (&acc)[8], bool bf16) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t keep = ((bits >> (2 * i)) & 1u ? 0x0000FFFFu : 0u) |
                          ((bits >> (2 * i + 1)) & 1u ? 0xFFFF0000u : 0u);
    w[i] &= keep;  // the select is on the bit pattern: +0 for both element types
    const float2 f = to_f32x2(bf16, w[i]);
    acc[2 * i] += f.x;
    acc[2 * i + 1] += f.y;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// dZ = dY * gelu'(z) for the eight 16-bit lanes of `v` (dY) and `z`; the fp32
// products are added to acc[0..7] before rounding.
__device__ __forceinline__ uint4 gelu_accumulate(uint4 v, uint4 z, float (&acc)[8], bool bf16) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const uint32_t zz[4] = {z.x, z.y, z.z, z.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 g = to_f32x2(bf16, w[i]);
    const float2 zf = to_f32x2(bf16, zz[i]);
    const float p0 = g.x * gelu_tanh_grad(zf.x);
    const float p1 = g.y * gelu_tanh_grad(zf.y);
    acc[2 * i] += p0;
    acc[2 * i + 1] += p1;
    o[i] = pack2(bf16, p0, p1);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// One 16-byte group (8 columns at c0 of row r) of either kind: mask bits
// (bits 0..7 of `bits`) or the pre-activations `z`.
template <bool GELU>
__device__ __forceinline__ uint4 apply_group(uint4 v, uint32_t bits, uint4 z, float (&acc)[8], bool bf16) {
  if constexpr (GELU)
    return gelu_accumulate(v, z, acc, bf16);
  else
    return mask_accumulate(v, bits, acc, bf16);
}

// Ragged element (column c of row r): the kept / scaled value and its fp32.
template <bool GELU>
__device__ __forceinline__ unsigned short apply_one(const DreluArgs& p, long long r, long long c,
                                                    unsigned short g, float& f, bool bf16) {
  if constexpr (GELU) {
    f = to_f32(bf16, g) * gelu_tanh_grad(to_f32(bf16, p.zaux[r * p.ld_zaux + c]));
    return from_f32(bf16, f);
  } else {
    const bool keep = (__ldg(p.mask + r * p.ld_aux + (c >> 5)) >> (c & 31)) & 1u;
    const unsigned short o = keep ? g : static_cast<unsigned short>(0);
    f = to_f32(bf16, o);
    return o;
  }
}

// DGELU_BGRAD keeps two blocks per SM: its derivative needs more registers.
template <bool GELU>
__global__ void __launch_bounds__(256, GELU ? 2 : MIN_BLOCKS) drelu_cols_kernel(const DreluArgs p) {
  constexpr int U = GELU ? UNROLL / 2 : UNROLL;  // the z loads double the registers in flight
  const bool bf16 = p.bf16 != 0;
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
      for (; r + (U - 1) * ROW_PHASES < r_end; r += U * ROW_PHASES) {
        uint4 v[U];
        uint32_t w[U];
        uint4 z[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const long long rr = r + u * ROW_PHASES;
          v[u] = ld_stream(p.dY + rr * p.ld + c0);
          if constexpr (GELU)
            z[u] = __ldg(reinterpret_cast<const uint4*>(p.zaux + rr * p.ld_zaux + c0));
          else
            w[u] = __ldg(p.mask + rr * p.ld_aux + widx);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const long long rr = r + u * ROW_PHASES;
          const uint4 o = apply_group<GELU>(v[u], w[u] >> bit_off, z[u], acc, bf16);
          st_stream(p.dZ + rr * p.ld + c0, o);
        }
      }
      for (; r < r_end; r += ROW_PHASES) {
        const uint4 v = ld_stream(p.dY + r * p.ld + c0);
        uint32_t w = 0;
        uint4 z = make_uint4(0, 0, 0, 0);
        if constexpr (GELU)
          z = __ldg(reinterpret_cast<const uint4*>(p.zaux + r * p.ld_zaux + c0));
        else
          w = __ldg(p.mask + r * p.ld_aux + widx);
        st_stream(p.dZ + r * p.ld + c0, apply_group<GELU>(v, w >> bit_off, z, acc, bf16));
      }
    } else {
      for (; r < r_end; r += ROW_PHASES) {  // ragged last strip: element-wise
        for (int j = 0; j < 8 && c0 + j < p.C; ++j) {
          const unsigned short g = reinterpret_cast<const unsigned short*>(p.dY)[r * p.ld + c0 + j];
          float f;
          reinterpret_cast<unsigned short*>(p.dZ)[r * p.ld + c0 + j] = apply_one<GELU>(p, r, c0 + j, g, f, bf16);
          acc[j] += f;
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

template <bool GELU>
__global__ void __launch_bounds__(256) drelu_rows_kernel(const DreluArgs p) {
  const bool bf16 = p.bf16 != 0;
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
    // RU 16-byte steps of the row per round: all their loads are issued
    // before any of their stores, so the round trips overlap.
    constexpr int RU = GELU ? 2 : 4;
    long long c = lane * 8;
    for (; c + (RU - 1) * 256 < C8; c += RU * 256) {
      uint4 v[RU], z[RU];
      uint32_t w[RU];
#pragma unroll
      for (int u = 0; u < RU; ++u) {
        const long long cc = c + u * 256;
        v[u] = ld_stream(src + cc);
        z[u] = make_uint4(0, 0, 0, 0);
        w[u] = 0;
        if constexpr (GELU)
          z[u] = __ldg(reinterpret_cast<const uint4*>(p.zaux + r * p.ld_zaux + cc));
        else
          w[u] = __ldg(mrow + (cc >> 5)) >> (cc & 31);
      }
#pragma unroll
      for (int u = 0; u < RU; ++u) st_stream(dst + c + u * 256, apply_group<GELU>(v[u], w[u], z[u], acc, bf16));
    }
    for (; c < C8; c += 256) {
      const uint4 v = ld_stream(src + c);
      uint32_t w = 0;
      uint4 z = make_uint4(0, 0, 0, 0);
      if constexpr (GELU)
        z = __ldg(reinterpret_cast<const uint4*>(p.zaux + r * p.ld_zaux + c));
      else
        w = __ldg(mrow + (c >> 5)) >> (c & 31);
      st_stream(dst + c, apply_group<GELU>(v, w, z, acc, bf16));
    }
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += acc[j];
    for (long long c = C8 + lane; c < p.C; c += 32) {  // ragged tail
      float f;
      reinterpret_cast<unsigned short*>(dst)[c] =
          apply_one<GELU>(p, r, c, reinterpret_cast<const unsigned short*>(src)[c], f, bf16);
      s += f;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) p.bgrad[r] = s;
  }
}

// out[i] = the sum over j of part[j * len + i] (the bias-gradient partials
// of a GEMM epilogue): a block takes 32 consecutive i, its 8 warps the rows
// j = w, w + 8, ... in order, and the first warp adds their 8 sums in warp
// order, so the result does not depend on timing. (A thread per i summing
// every row in turn kept too few loads in flight: 256 partial rows of 11008
// took tens of microseconds.)
__global__ void __launch_bounds__(256) bgrad_reduce_kernel(const float* part, long long rows, long long len,
                                                           float* out) {
  __shared__ float red[8][32];
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  for (long long c0 = blockIdx.x * 32LL; c0 < len; c0 += gridDim.x * 32LL) {
    const long long i = c0 + lane;
    float s = 0.0f;
    if (i < len) {
      long long j = w;
      for (; j + 24 < rows; j += 32) {  // four rows of this warp's share per step
        const float a0 = __ldcg(part + j * len + i);
        const float a1 = __ldcg(part + (j + 8) * len + i);
        const float a2 = __ldcg(part + (j + 16) * len + i);
        const float a3 = __ldcg(part + (j + 24) * len + i);
        s += a0;
        s += a1;
        s += a2;
        s += a3;
      }
      for (; j < rows; j += 8) s += __ldcg(part + j * len + i);
    }
    red[w][lane] = s;
    __syncthreads();
    if (w == 0 && i < len) {
      float t = 0.0f;
#pragma unroll
      for (int k = 0; k < 8; ++k) t += red[k][lane];
      out[i] = t;
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_bgrad_reduce(const float* part, long long rows, long long len, float* out,
                                cudaStream_t stream) {
  if (len <= 0) return cudaSuccess;
  long long blocks = (len + 31) / 32;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  bgrad_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(part, rows, len, out);
  return cudaGetLastError();
}

// Row splits for the column case: one wave of resident blocks (measured on
// dY[8192, 11008], 43 strips, 3 blocks per SM: 8 or 10 splits (0.75 and 0.94
// waves) take 58 us, 12 splits (1.13 waves) 75 us, 15 and 18 splits 65 and
// 62 us), at least 64 rows per split, at most 256 splits. GE_DRELU_SPLITS
// overrides (sweeps).
int drelu_splits(long long R, long long C, int num_sms, int gelu) {
  static std::atomic<int> occ[2] = {0, 0};
  if (occ[gelu ? 1 : 0] == 0) {
    int o = 0;
    const cudaError_t e =
        gelu ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, drelu_cols_kernel<true>, 256, 0)
             : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, drelu_cols_kernel<false>, 256, 0);
    if (e != cudaSuccess || o < 1) {
      cudaGetLastError();
      o = gelu ? 2 : MIN_BLOCKS;
    }
    occ[gelu ? 1 : 0] = o;
  }
  const int occupancy = occ[gelu ? 1 : 0];
  const long long strips = (C + COLS_PER_BLOCK - 1) / COLS_PER_BLOCK;
  // One wave: the largest split count whose blocks are all resident at once.
  // A partly filled second wave leaves most SMs idle while its blocks run.
  long long want = static_cast<long long>(occupancy) * num_sms / strips;
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
    if (a.gelu)
      drelu_cols_kernel<true><<<grid, 256, 0, s>>>(a);
    else
      drelu_cols_kernel<false><<<grid, 256, 0, s>>>(a);
  } else {
    long long blocks = (a.R + 7) / 8;
    if (blocks > 65535LL * 16) blocks = 65535LL * 16;
    if (a.gelu)
      drelu_rows_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
    else
      drelu_rows_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace ge
