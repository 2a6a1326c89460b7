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
// Streaming kernel (N <= 4, K <= 8192): one CTA per SM owns a contiguous
// share of the weight rows; one producer lane first bulk-copies the N
// activation vectors into shared memory, then keeps a shared-memory ring of
// whole weight rows full with 1-D bulk copies (TMA), about 64 KB per SM
// in flight; eight consumer warps (warp w owns ring slots w, w+8, ...) read
// rows and activations from shared memory with 16-byte loads, accumulate in
// fp32, reduce across the warp and apply bias + activation + fp16 rounding.
// Every wait is bounded (error word, then drain and exit).
// Other shapes use the register kernel below: one warp per row, 16-byte
// non-allocating global loads, UNROLL slabs in flight.
#include <cstdlib>

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
  {
    // Ask L2 for this warp's first weight row before waiting on the previous
    // grid (with programmatic dependent launch that grid may still run).
    const long long m0 = blockIdx.x * wpb + (threadIdx.x >> 5);
    if (lane == 0 && m0 < p.M && (p.K & 7) == 0)
      bulk_prefetch_l2(p.A + m0 * p.lda, static_cast<uint32_t>(p.K) * 2u);
  }
  grid_launch_dependents();
  grid_dependency_wait();  // B may come from, and D may be read by, the previous grid
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
      else if (p.epi == EPI_GELU_ERF_BIAS) y = gelu_erf(z);
      p.D[m * p.ldd_m + static_cast<long long>(lane) * p.ldd_n] = __float2half_rn(y);
    }
  }
}

constexpr int GV_WARPS = 8;                    // consumer warps
constexpr int GV_THREADS = 32 * (GV_WARPS + 1);  // + one producer warp
constexpr int GV_RING_BYTES = 200 * 1024;
constexpr int GV_SLOTS = 8;  // rows in flight per CTA

__device__ __forceinline__ float gemv_act(int epi, float z) {
  if (epi == EPI_RELU_BIAS) return fmaxf(z, 0.0f);
  if (epi == EPI_GELU_BIAS) return gelu_tanh(z);
  if (epi == EPI_GELU_ERF_BIAS) return gelu_erf(z);
  return z;
}

template <int NT>
__global__ void __launch_bounds__(GV_THREADS, 1)
    gemv_stream_kernel(const GemvArgs p, int slots, uint32_t slot_bytes, uint32_t x_stride_bytes) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // [full[slots] | empty[slots] | xbar | abort, never] [x: N rows of K fp16]
  // [ring of weight rows]; x and the ring start on 128-byte boundaries.
  const uint32_t bar0 = smem_u32(smem);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (slots + s); };
  const uint32_t x_bar = bar0 + 16u * slots;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 16 * slots + 8);
  volatile int* never = abort_flag + 1;
  const uint32_t x_off = (16u * slots + 16u + 127u) & ~127u;
  const __half* xs = reinterpret_cast<const __half*>(smem + x_off);
  uint8_t* ring = smem + x_off + static_cast<uint32_t>(p.N) * x_stride_bytes;
  const uint32_t row_bytes = static_cast<uint32_t>(p.K) * 2u;  // K % 8 == 0
  const int x_stride = static_cast<int>(x_stride_bytes / 2);

  // Contiguous, balanced share of rows for this CTA.
  const long long per = p.M / gridDim.x;
  const long long extra = p.M % gridDim.x;
  const long long r0 = blockIdx.x * per + min(static_cast<long long>(blockIdx.x), extra);
  const long long nr = per + (static_cast<long long>(blockIdx.x) < extra ? 1 : 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < slots; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(x_bar, 1);
    *abort_flag = 0;
    *never = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == GV_WARPS) {
    if (lane == 0) {
      // The first ring's worth of weight rows are requested before waiting
      // for the previous grid on the stream (with programmatic dependent
      // launch that grid may still be running; A is static by contract).
      long long issued = 0;
      const long long first = nr < slots ? nr : slots;
      for (long long j = 0; j < first; ++j) {
        mbar_arrive_expect_tx(full_bar(static_cast<int>(j)), row_bytes);
        bulk_load_1d(smem_u32(ring + static_cast<size_t>(j) * slot_bytes), p.A + (r0 + j) * p.lda,
                     row_bytes, full_bar(static_cast<int>(j)));
        ++issued;
      }
      grid_launch_dependents();
      grid_dependency_wait();  // the activations may come from the previous grid
      mbar_arrive_expect_tx(x_bar, static_cast<uint32_t>(p.N) * row_bytes);
      for (int n = 0; n < p.N; ++n)
        bulk_load_1d(smem_u32(smem + x_off) + static_cast<uint32_t>(n) * x_stride_bytes,
                     p.B + n * p.ldb, row_bytes, x_bar);
      for (long long j = first; j < nr; ++j) {
        const int s = static_cast<int>(j % slots);
        const uint32_t ph = static_cast<uint32_t>((j / slots) & 1);
        if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, p.budget)) {
          if (!*abort_flag) atomicOr(p.err, ERR_GEMV_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(full_bar(s), row_bytes);
        bulk_load_1d(smem_u32(ring + static_cast<size_t>(s) * slot_bytes), p.A + (r0 + j) * p.lda,
                     row_bytes, full_bar(s));
        ++issued;
      }
      // Drain: every issued copy lands before the CTA may exit.
      if (!mbar_wait_bounded(x_bar, 0u, never, p.budget)) atomicOr(p.err, ERR_GEMV_TIMEOUT);
      for (long long j = issued - slots > 0 ? issued - slots : 0; j < issued; ++j) {
        const int s = static_cast<int>(j % slots);
        if (!mbar_wait_bounded(full_bar(s), static_cast<uint32_t>((j / slots) & 1), never, p.budget))
          atomicOr(p.err, ERR_GEMV_TIMEOUT);
      }
    }
  } else {
    grid_dependency_wait();  // D may still be read by the previous grid
    int ok = 1;
    if (lane == 0) ok = mbar_wait_bounded(x_bar, 0u, abort_flag, p.budget) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok && lane == 0) {
      if (!*abort_flag) atomicOr(p.err, ERR_GEMV_TIMEOUT);
      *abort_flag = 1;
    }
    // Every slot is consumed by one warp only (slot s by warp s % GV_WARPS),
    // row after row in fill order, so a warp never waits on a parity two
    // phases ahead of the barrier (which would alias the completed phase).
    for (long long j = 0; ok && j < nr; ++j) {
      const int s = static_cast<int>(j % slots);
      if (s % GV_WARPS != warp) continue;
      const uint32_t ph = static_cast<uint32_t>((j / slots) & 1);
      if (lane == 0) ok = mbar_wait_bounded(full_bar(s), ph, abort_flag, p.budget) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) {
          if (!*abort_flag) atomicOr(p.err, ERR_GEMV_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      const __half* row = reinterpret_cast<const __half*>(ring + static_cast<size_t>(s) * slot_bytes);
      float acc[NT];
#pragma unroll
      for (int n = 0; n < NT; ++n) acc[n] = 0.0f;
#pragma unroll 4
      for (int k = lane * 8; k < p.K; k += 256) {
        const uint4 a = *reinterpret_cast<const uint4*>(row + k);
#pragma unroll
        for (int n = 0; n < NT; ++n)
          if (n < p.N) acc[n] = dot8(a, *reinterpret_cast<const uint4*>(xs + n * x_stride + k), acc[n]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));  // the row is in registers now
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
        const long long m = r0 + j;
        if (p.epi != EPI_NONE) z += __half2float(p.bias[m]);
        p.D[m * p.ldd_m + static_cast<long long>(lane) * p.ldd_n] = __float2half_rn(gemv_act(p.epi, z));
      }
    }
  }
}

template <int NT>
cudaError_t launch_stream(const GemvArgs& a, int num_sms, cudaStream_t s) {
  const uint32_t row_bytes = static_cast<uint32_t>(a.K) * 2u;
  const uint32_t slot_bytes = (row_bytes + 127u) & ~127u;
  const uint32_t x_stride_bytes = slot_bytes;
  const int grid = static_cast<int>(a.M < num_sms ? a.M : num_sms);
  const long long rows_max = (a.M + grid - 1) / grid;
  const uint32_t x_bytes = static_cast<uint32_t>(a.N) * x_stride_bytes;
  // Up to GV_SLOTS rows in flight per SM: more outstanding copies than that
  // measured slower (12.3 us with 24 x 8 KB per SM vs 10.3 us with 6-12 for a
  // 33.5 MB weight), so the ring is sized for ~64 KB in flight, a multiple of
  // the consumer-warp count when the ring has to wrap.
  int slots = static_cast<int>((GV_RING_BYTES - x_bytes) / slot_bytes);
  if (slots > GV_SLOTS) slots = GV_SLOTS;
  if (slots > rows_max) slots = static_cast<int>(rows_max);
  if (slots < 1) slots = 1;
  const size_t smem = ((16u * slots + 16u + 127u) & ~127u) + x_bytes + static_cast<size_t>(slots) * slot_bytes;
  static bool configured[64] = {};  // the attribute is set once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(gemv_stream_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             GV_RING_BYTES + 1024);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(GV_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (a.static_a) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  e = cudaLaunchKernelEx(&cfg, gemv_stream_kernel<NT>, a, slots, slot_bytes, x_stride_bytes);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int NT, int UNROLL>
cudaError_t launch_nt(const GemvArgs& a, int num_sms, cudaStream_t s) {
  constexpr int threads = 256;
  long long blocks = (a.M + 7) / 8;  // one row per warp when the grid allows
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (a.static_a) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_kernel<NT, UNROLL>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const GemvArgs& a, int num_sms, cudaStream_t s) {
  // The streaming kernel wants whole rows in the ring (K <= 8192), rows that
  // are a whole number of 16-byte chunks (K % 8 == 0) starting on 16-byte
  // boundaries (the planner checks lda % 8 == 0 and A's alignment), and
  // activations small enough to stay in L1 (N <= 4).
  // GE_GEMV_KERNEL=stream|reg selects the kernel (A/B measurements).
  bool stream_ok = a.K <= 8192 && a.K % 8 == 0 && a.N <= 4 && a.M >= 1;
  if (const char* env = std::getenv("GE_GEMV_KERNEL")) {
    if (env[0] == 'r') stream_ok = false;
  }
  if (stream_ok) {
    if (a.N <= 1) return launch_stream<1>(a, num_sms, s);
    if (a.N <= 2) return launch_stream<2>(a, num_sms, s);
    return launch_stream<4>(a, num_sms, s);
  }
  if (a.N <= 1) return launch_nt<1, 8>(a, num_sms, s);
  if (a.N <= 2) return launch_nt<2, 8>(a, num_sms, s);
  if (a.N <= 4) return launch_nt<4, 4>(a, num_sms, s);
  if (a.N <= 8) return launch_nt<8, 4>(a, num_sms, s);
  return launch_nt<16, 2>(a, num_sms, s);
}

}  // namespace ge
