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
// With static weights the plan launches the kernel as a programmatic
// dependent, so a chain of decode projections starts layer i+1's weight reads
// while layer i drains: for N = 1 (fp16) each warp loads the first half of
// its row into registers before it waits for the previous grid (back to back
// over 8 weights of 4096 x 4096: 9.8 -> 8.0 us a layer), then the rest in
// one 8-slab round; for larger N, with fewer slabs in flight per warp, each
// warp first asks L2 for its first row with one bulk prefetch (PF). For
// N = 1 a warp issues a whole 4096-element row (16 slabs) at once.
//
// For every N the grid is one block per SM of ceil(M / SMs) warps (4 to
// 27): 4096 rows are 152 blocks of 27 warps, every row's loads issued by
// the first wave of blocks. Measured against the earlier shapes (4-warp
// blocks for N = 1, 8-warp blocks otherwise; same GPU, alternating runs, L2
// flushed), single launches: 4096 x 4096 N = 1 12.9 us either way (the old
// shape 15.0 in some runs), back to back 7.6 against 8.0 us a layer; N = 2
// 17.0 against 19.1 us, N = 4 25.2 either way, N = 8 33.4 against 40, N = 16
// 86.7 against 119; N = 1 on 11008 x 4096 23.2 against 27.3 us and on
// 16384 x 4096 27.4-29.3 against 33.4-35.5 us. Earlier N = 1 forms: 14-warp
// blocks 15.0 / 7.7 us; 8 slabs, 8-warp blocks, prefetch 14.5 / 8.8 us; 16
// slabs with the prefetch 15.9 / 10.3 us. (A variant that streamed rows
// through a shared-memory ring with bulk copies measured slower still: 11.8
// us per layer back to back.)
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

// BF16 picks the element type of A, B, bias and D at compile time so that the
// fp16 and bf16 inner loops each decode with one instruction per pair.
constexpr int kGemvMaxWarps = 27;  // warps a block at most (the launch bound)

template <int NT, int UNROLL, bool BF16, bool PF, bool PRE = false>
__global__ void __launch_bounds__(32 * kGemvMaxWarps) gemv_kernel(const GemvArgs p) {
  const int lane = threadIdx.x & 31;
  const long long wpb = blockDim.x >> 5;
  const long long nwarps = static_cast<long long>(gridDim.x) * wpb;
  const int K8 = p.K & ~7;
  constexpr int SLAB = 32 * 8;  // elements one warp covers per 16-byte load
  if (PF) {
    // Ask L2 for this warp's first weight row before waiting on the previous
    // grid (with programmatic dependent launch that grid may still run).
    const long long m0 = blockIdx.x * wpb + (threadIdx.x >> 5);
    if (lane == 0 && m0 < p.M && (p.K & 7) == 0)
      bulk_prefetch_l2(p.A + m0 * p.lda, static_cast<uint32_t>(p.K) * 2u);
  }
  // PRE (static weights): the first PRE_SLABS slabs of this warp's first
  // row are requested before the wait on the previous grid, which may still
  // be running, so a chain of decode projections streams weights across
  // layer boundaries. fp16 only: the bf16 decode needs more registers per
  // slab, and with the preload a 4096-row grid no longer fits at once
  // (measured 13.2 -> 19.6 us for one launch).
  constexpr bool PRELOAD = PRE && !BF16;
  constexpr int PRE_SLABS = 8;
  const long long m_first = blockIdx.x * wpb + (threadIdx.x >> 5);
  uint4 pre[PRELOAD ? PRE_SLABS : 1];
  bool have_pre = false;
  if constexpr (PRELOAD) {
    if (p.static_a && m_first < p.M && lane * 8 + (PRE_SLABS - 1) * SLAB < K8) {
      const __half* arow = p.A + m_first * p.lda;
#pragma unroll
      for (int u = 0; u < PRE_SLABS; ++u) pre[u] = ld_stream(arow + lane * 8 + u * SLAB);
      have_pre = true;
    }
  }
  grid_launch_dependents();
  grid_dependency_wait();  // B may come from, and D may be read by, the previous grid
  for (long long m = m_first; m < p.M; m += nwarps) {
    const __half* arow = p.A + m * p.lda;
    if (lane == 0 && p.err) (void)GE_DCHECK(m >= 0 && p.K <= p.lda && p.N <= NT, p.err);
    float acc[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n] = 0.0f;
    int k = lane * 8;
    if constexpr (PRELOAD) {
      if (have_pre && m == m_first) {
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          if (n < p.N) {
            const __half* brow = p.B + n * p.ldb + k;
#pragma unroll
            for (int u = 0; u < PRE_SLABS; ++u)
              acc[n] = dot8<BF16>(pre[u], __ldg(reinterpret_cast<const uint4*>(brow + u * SLAB)), acc[n]);
          }
        }
        k += PRE_SLABS * SLAB;
      }
    }
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
            acc[n] = dot8<BF16>(a[u], __ldg(reinterpret_cast<const uint4*>(brow + u * SLAB)), acc[n]);
        }
      }
    }
    if constexpr (UNROLL > 4) {  // what is left of the row, MID slabs at a time
      constexpr int MID = UNROLL >= 16 ? 8 : 4;
      for (; k + (MID - 1) * SLAB < K8; k += MID * SLAB) {
        uint4 a[MID];
#pragma unroll
        for (int u = 0; u < MID; ++u) a[u] = ld_stream(arow + k + u * SLAB);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          if (n < p.N) {
            const __half* brow = p.B + n * p.ldb + k;
#pragma unroll
            for (int u = 0; u < MID; ++u)
              acc[n] = dot8<BF16>(a[u], __ldg(reinterpret_cast<const uint4*>(brow + u * SLAB)), acc[n]);
          }
        }
      }
    }
    for (; k < K8; k += SLAB) {
      const uint4 a = ld_stream(arow + k);
#pragma unroll
      for (int n = 0; n < NT; ++n)
        if (n < p.N) acc[n] = dot8<BF16>(a, __ldg(reinterpret_cast<const uint4*>(p.B + n * p.ldb + k)), acc[n]);
    }
    for (int kk = K8 + lane; kk < p.K; kk += 32) {  // ragged K tail
      const float av = to_f32(BF16, reinterpret_cast<const unsigned short*>(arow)[kk]);
#pragma unroll
      for (int n = 0; n < NT; ++n)
        if (n < p.N)
          acc[n] = fmaf(av, to_f32(BF16, reinterpret_cast<const unsigned short*>(p.B)[n * p.ldb + kk]), acc[n]);
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
      if (p.epi != EPI_NONE) z += to_f32(BF16, reinterpret_cast<const unsigned short*>(p.bias)[m]);
      if (p.epi == EPI_BIAS_RESIDUAL)
        z += to_f32(BF16, p.res[m * p.ldd_m + static_cast<long long>(lane) * p.ldd_n]);
      float y = z;
      if (p.epi == EPI_RELU_BIAS) y = fmaxf(z, 0.0f);
      else if (p.epi == EPI_GELU_BIAS) y = gelu_tanh(z);
      else if (p.epi == EPI_GELU_ERF_BIAS) y = gelu_erf(z);
      reinterpret_cast<unsigned short*>(p.D)[m * p.ldd_m + static_cast<long long>(lane) * p.ldd_n] =
          from_f32(BF16, y);
    }
  }
}

template <int NT, int UNROLL, bool PF, bool PRE = false>
cudaError_t launch_nt(const GemvArgs& a, int num_sms, cudaStream_t s) {
  // one block per SM of ceil(M / SMs) warps (4 to kGemvMaxWarps), one row
  // per warp when the grid allows (warps stride over the rest)
  const long long w = (a.M + num_sms - 1) / num_sms;
  const long long warps = w < 4 ? 4 : (w > kGemvMaxWarps ? kGemvMaxWarps : w);
  long long blocks = (a.M + warps - 1) / warps;
  if (blocks > num_sms) blocks = num_sms;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(32 * warps), 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (a.static_a) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cudaError_t e = a.bf16 ? cudaLaunchKernelEx(&cfg, gemv_kernel<NT, UNROLL, true, PF, PRE>, a)
                         : cudaLaunchKernelEx(&cfg, gemv_kernel<NT, UNROLL, false, PF, PRE>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const GemvArgs& a, int num_sms, cudaStream_t s) {
  if (a.N <= 1) return launch_nt<1, 16, false, true>(a, num_sms, s);
  if (a.N <= 2) return launch_nt<2, 8, true>(a, num_sms, s);
  if (a.N <= 4) return launch_nt<4, 4, true>(a, num_sms, s);
  if (a.N <= 8) return launch_nt<8, 4, true>(a, num_sms, s);
  return launch_nt<16, 2, true>(a, num_sms, s);
}

}  // namespace ge
