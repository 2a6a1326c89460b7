// ge_chain.cu -- a stack of decode projections in one persistent launch.
//
// ops-nn MatMul fusion (codearts), "Why MatMul is the inference bottleneck":
// a decode step carries one token's activations through one weight matrix
// after another, and each layer costs the time to read its weights once from
// HBM; the bias and activation ride along in the epilogue ("ops-nn's MatMul
// fusion strategy", first level). Launched one layer at a time, every layer
// also pays a launch, a ramp-up and a drain during which HBM idles. Here one
// cooperative launch runs all the layers. The weights do not depend on the
// activations, so every warp keeps streaming its next weight rows -- of this
// layer and of the following ones -- into shared memory while the grid waits
// for the previous layer's outputs.
//
// Work split: one block per SM of CW warps (16 for up to four tokens, the
// weight rows then cut in two segments; 8 with whole rows otherwise). Block b
// owns rows [b*M/G, (b+1)*M/G) of every layer (G blocks), warp w of the
// block the rows r0 + w + CW*j. A warp's work is the sequence of its row
// segments, layer after layer; item t of that sequence lands in the warp's
// own ring slot t % R (R segment-sized slots), filled by lane 0 with one 1-D
// bulk copy counted on the slot's mbarrier. The warp consumes its items in
// order and refills a slot only after it consumed it, so a slot's barrier
// never runs a phase ahead of its waiter and no other warp touches the slot.
// Per layer: the block waits until every block has stored layer l-1 (one
// counter per layer: release add by each block, acquire load by the
// waiter), stages the N x K activations in shared memory, and then, for each
// of its items: wait for the slot, fp32 dot products from shared memory,
// refill the slot; after a row's last segment, butterfly reduction, bias +
// activation, round, store. Every wait is bounded: an expired wait sets
// ERR_CHAIN_TIMEOUT and a grid-wide abort flag, and every warp waits
// (bounded) for its copies in flight before the block exits. The last block
// to finish clears the counters and the flag for the next launch.
//
// Measured on 32 layers of 4096 x 4096 fp16, one token (one launch, L2
// flushed): 8.3-8.7 us a layer. A read-only stream of the same bytes through
// the same ring (no layer dependence) reaches 6.8-7.1 TB/s, i.e. 4.7 us a
// layer: the gap is the wait at every layer boundary, during which the ring
// (192 KB per SM) is full of the next layer's rows (216 KB per SM per layer)
// and HBM idles. Requesting the layers ahead into L2 with bulk prefetches
// measured slower (1, 2, 3 or 4 layers ahead: +11-15 %), and so did backing
// off the counter polls, 32 warps with quarter-row items, and keeping one
// token's activations in registers (every warp then reads them from L2).
#include <atomic>

#include "ge_internal.h"
#include "ge_ptx.cuh"

namespace ge {
namespace {

constexpr int kSmemMax = 232448;        // dynamic shared memory per block
constexpr int kSmemSlack = 128 + 16;    // base alignment + the block's flags

__device__ __forceinline__ float chain_act(int epi, float z) {
  if (epi == EPI_RELU_BIAS) return fmaxf(z, 0.0f);
  if (epi == EPI_GELU_BIAS) return gelu_tanh(z);
  if (epi == EPI_GELU_ERF_BIAS) return gelu_erf(z);
  return z;
}

size_t x_bytes(int K, int N) { return (static_cast<size_t>(N) * K * 2 + 127) & ~static_cast<size_t>(127); }

// Launch shape: warps per block and segments per weight row (one ring item
// is one segment). Wide rows of few tokens take 16 warps and half-row items:
// twice the rows in progress at once, the same bytes in flight.
struct Shape {
  int warps, seg;
};
Shape chain_shape(int K, int N) {
  if (N <= 4 && K % 16 == 0) return {16, 2};
  return {8, 1};
}

int ring_for(int K, int N, Shape sh) {
  const long long seg_bytes = 2LL * K / sh.seg;
  const long long avail = kSmemMax - kSmemSlack - static_cast<long long>(x_bytes(K, N));
  long long r = avail > 0 ? avail / (sh.warps * (seg_bytes + 8)) : 0;
  if (r > 8) r = 8;
  return static_cast<int>(r);
}

size_t chain_smem(int K, int N, Shape sh, int ring) {
  return kSmemSlack + x_bytes(K, N) + static_cast<size_t>(sh.warps) * ring * (2ull * K / sh.seg + 8);
}

template <int NT, bool BF16, int CW, int SEG>
__global__ void __launch_bounds__(32 * CW, 1) gemv_chain_kernel(const __grid_constant__ ChainArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t row_bytes = static_cast<uint32_t>(p.K) * 2u;
  const uint32_t seg_bytes = row_bytes / SEG;
  const int C16 = (p.K >> 3) / SEG;  // 16-byte chunks per segment
  const size_t xb = (static_cast<size_t>(p.N) * row_bytes + 127) & ~static_cast<size_t>(127);
  uint8_t* xs = smem;
  uint8_t* rings = smem + xb;
  uint8_t* ring = rings + static_cast<size_t>(warp) * p.ring * seg_bytes;
  const uint32_t ring_s = smem_u32(ring);
  uint8_t* bars = rings + static_cast<size_t>(CW) * p.ring * seg_bytes;
  const uint32_t bar0 = smem_u32(bars) + 8u * static_cast<uint32_t>(warp * p.ring);
  volatile int* abort_s = reinterpret_cast<volatile int*>(bars + 8 * CW * p.ring);
  volatile int* never = abort_s + 1;
  unsigned int* const counters = p.sync;
  unsigned int* const done = p.sync + kChainMaxLayers;
  volatile unsigned int* const abort_g = p.sync + kChainMaxLayers + 1;

  const int r0 = static_cast<int>(static_cast<long long>(blockIdx.x) * p.M / gridDim.x);
  const int r1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * p.M / gridDim.x);
  const int nrw = r1 - r0 > warp ? (r1 - r0 - warp + CW - 1) / CW : 0;  // rows of this warp per layer
  const int per_layer = nrw * SEG;                                       // items of this warp per layer
  const long long total = static_cast<long long>(per_layer) * p.layers;

  if (lane == 0)
    for (int s = 0; s < p.ring; ++s) mbar_init(bar0 + 8u * s, 1);
  if (threadIdx.x == 0) {
    *abort_s = 0;
    *never = 0;
  }
  fence_barrier_init();
  __syncthreads();

  // item t: layer t / per_layer; within it row j = (t % per_layer) / SEG
  // (global row r0 + warp + CW * j), segment h = t % SEG; ring slot t % ring
  auto issue = [&](long long t) {
    const int l = static_cast<int>(t / per_layer);
    const int q = static_cast<int>(t - static_cast<long long>(l) * per_layer);
    const long long row = r0 + warp + CW * (q / SEG);
    const int s = static_cast<int>(t % p.ring);
    const uint32_t bar = bar0 + 8u * s;
    // (GE_DEBUG) the item lies in this warp's sequence, its row in the
    // block's range, its slot in the warp's ring; a skipped copy ends in
    // the consumer's bounded wait
    if (!GE_DCHECK(t >= 0 && t < total && l < p.layers && row < r1 && s < p.ring, p.err)) return;
    mbar_arrive_expect_tx(bar, seg_bytes);
    bulk_load_1d(ring_s + static_cast<uint32_t>(s) * seg_bytes,
                 reinterpret_cast<const uint8_t*>(p.A[l] + row * p.lda) + (q % SEG) * seg_bytes, seg_bytes, bar);
  };
  long long issued = 0;  // lane 0's count of items whose copies were issued
  if (lane == 0)
    for (; issued < total && issued < p.ring; ++issued) issue(issued);

  long long t = 0;  // items consumed (the same in every lane)
  for (int l = 0; l < p.layers; ++l) {
    // The bias of this warp's rows of the layer, requested before the wait
    // for the previous layer: lane j holds row j's (the first 32 rows); kept
    // as loaded and converted at use, so nothing waits on it here.
    const unsigned short* bias = p.bias[l];
    unsigned short braw = 0;
    if (p.epi != EPI_NONE && lane < nrw) braw = bias[r0 + warp + CW * lane];
    if (l > 0) {
      // every block has stored layer l - 1
      if (threadIdx.x == 0) {
        const long long t0 = clock64();
        while (ld_acquire_gpu(counters + (l - 1)) < gridDim.x) {
          if (*abort_g != 0) {
            *abort_s = 1;
            break;
          }
          if (clock64() - t0 > p.budget) {
            atomicOr(p.err, ERR_CHAIN_TIMEOUT);
            *abort_g = 1;
            *abort_s = 1;
            break;
          }
        }
      }
      __syncthreads();
      if (*abort_s) break;
    }
    // this layer's activations: X, or the previous layer's stored outputs
    const unsigned short* xsrc = l == 0 ? p.X : p.Y + static_cast<long long>(l - 1) * p.N * p.ldy;
    const long long xld = l == 0 ? p.ldx : p.ldy;
    const int K16 = p.K >> 3;
    for (int i = threadIdx.x; i < p.N * K16; i += blockDim.x) {
      const int n = i / K16;
      const int c = i - n * K16;
      *reinterpret_cast<uint4*>(xs + static_cast<size_t>(n) * row_bytes + 16 * c) = ld_cg_u4(xsrc + n * xld + 8 * c);
    }
    __syncthreads();
    unsigned short* ydst = p.Y + static_cast<long long>(l) * p.N * p.ldy;
    // two accumulators per token (alternate 16-byte chunks) halve the chain
    // of dependent multiply-adds; added in a fixed order at the row's end
    float acc[NT], acc2[NT];
    for (int q = 0; q < per_layer; ++q) {
      if (__any_sync(0xffffffffu, *abort_s != 0)) break;  // the same decision in every lane
      const int j = q / SEG, h = q % SEG;
      const int s = static_cast<int>(t % p.ring);
      // (GE_DEBUG) lane 0 issues at most `ring` items ahead of the ones
      // consumed: a slot's barrier is never a phase ahead of its waiter
      if (lane == 0) (void)GE_DCHECK(issued - t <= p.ring && issued >= t, p.err);
      const uint32_t par = static_cast<uint32_t>((t / p.ring) & 1);
      const bool landed = mbar_wait_bounded(bar0 + 8u * s, par, abort_s, p.budget);
      if (!__all_sync(0xffffffffu, landed)) {
        if (lane == 0 && !*abort_s) {
          atomicOr(p.err, ERR_CHAIN_TIMEOUT);
          *abort_g = 1;
          *abort_s = 1;
        }
        break;
      }
      const uint8_t* wseg = ring + static_cast<size_t>(s) * seg_bytes;
      const uint8_t* xseg = xs + static_cast<size_t>(h) * seg_bytes;
      if (h == 0) {
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[n] = acc2[n] = 0.0f;
      }
      int c = lane;
      for (; c + 32 < C16; c += 64) {
        const uint4 w0 = *reinterpret_cast<const uint4*>(wseg + 16 * c);
        const uint4 w1 = *reinterpret_cast<const uint4*>(wseg + 16 * (c + 32));
#pragma unroll
        for (int n = 0; n < NT; ++n)
          if (n < p.N) {
            const uint8_t* xr = xseg + static_cast<size_t>(n) * row_bytes;
            acc[n] = dot8<BF16>(w0, *reinterpret_cast<const uint4*>(xr + 16 * c), acc[n]);
            acc2[n] = dot8<BF16>(w1, *reinterpret_cast<const uint4*>(xr + 16 * (c + 32)), acc2[n]);
          }
      }
      if (c < C16) {
        const uint4 w0 = *reinterpret_cast<const uint4*>(wseg + 16 * c);
#pragma unroll
        for (int n = 0; n < NT; ++n)
          if (n < p.N)
            acc[n] = dot8<BF16>(w0, *reinterpret_cast<const uint4*>(xseg + static_cast<size_t>(n) * row_bytes + 16 * c),
                                acc[n]);
      }
      ++t;
      __syncwarp();
      // the slot is consumed: it takes the warp's next item (its shared-memory
      // reads are ordered before the bulk copy's writes)
      if (lane == 0 && issued < total) {
        fence_proxy_async_smem();
        issue(issued);
        ++issued;
      }
      if (h != SEG - 1) continue;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        acc[n] += acc2[n];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc[n] += __shfl_xor_sync(0xffffffffu, acc[n], off);
      }
      float z = 0.0f;
#pragma unroll
      for (int n = 0; n < NT; ++n)
        if (n == lane) z = acc[n];
      const unsigned short bj = j < 32 ? static_cast<unsigned short>(__shfl_sync(0xffffffffu, braw, j)) : 0;
      if (lane < p.N) {
        const long long row = r0 + warp + CW * j;
        if (p.epi != EPI_NONE) z += to_f32(BF16, j < 32 ? bj : bias[row]);
        ydst[static_cast<long long>(lane) * p.ldy + row] = from_f32(BF16, chain_act(p.epi, z));
      }
    }
    __syncthreads();
    if (*abort_s) break;
    // this block's rows of layer l are stored
    if (threadIdx.x == 0) {
      __threadfence();
      red_release_gpu_add(counters + l, 1u);
    }
  }

  // After an abort, copies may still be in flight into this warp's slots:
  // they must land before the block's shared memory goes away.
  if (lane == 0) {
    for (long long u = t; u < issued; ++u) {
      const int s = static_cast<int>(u % p.ring);
      const uint32_t par = static_cast<uint32_t>((u / p.ring) & 1);
      if (!mbar_wait_bounded(bar0 + 8u * s, par, never, p.budget)) atomicOr(p.err, ERR_DRAIN_TIMEOUT);
    }
  }
  __syncthreads();
  // The last block to get here is past every wait of every block: it clears
  // the counters and the abort flag for the next launch.
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned int prev = atomicAdd(done, 1u);
    if (prev == gridDim.x - 1) {
      for (int l = 0; l < p.layers; ++l) counters[l] = 0u;
      *abort_g = 0u;
      __threadfence();
      atomicExch(done, 0u);
    }
  }
}

template <int NT, bool BF16, int CW, int SEG>
cudaError_t launch_chain_t(const ChainArgs& a, int num_sms, cudaStream_t s) {
  static std::atomic<bool> configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(gemv_chain_kernel<NT, BF16, CW, SEG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemMax);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  const size_t smem = chain_smem(a.K, a.N, Shape{CW, SEG}, a.ring);
  // The blocks wait on one another: all of them must be resident at once,
  // which the cooperative launch guarantees (or refuses).
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_chain_kernel<NT, BF16, CW, SEG>, 32 * CW, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms), 1, 1);
  cfg.blockDim = dim3(32 * CW, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gemv_chain_kernel<NT, BF16, CW, SEG>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int NT>
cudaError_t launch_chain_nt(const ChainArgs& a, int num_sms, cudaStream_t s) {
  const Shape sh = chain_shape(a.K, a.N);
  if constexpr (NT <= 4) {
    if (sh.warps == 16)
      return a.bf16 ? launch_chain_t<NT, true, 16, 2>(a, num_sms, s) : launch_chain_t<NT, false, 16, 2>(a, num_sms, s);
  }
  return a.bf16 ? launch_chain_t<NT, true, 8, 1>(a, num_sms, s) : launch_chain_t<NT, false, 8, 1>(a, num_sms, s);
}

}  // namespace

int gemv_chain_ring(int K, int N) { return ring_for(K, N, chain_shape(K, N)); }

cudaError_t launch_gemv_chain(const ChainArgs& a, int num_sms, cudaStream_t s) {
  if (a.N <= 1) return launch_chain_nt<1>(a, num_sms, s);
  if (a.N <= 2) return launch_chain_nt<2>(a, num_sms, s);
  if (a.N <= 4) return launch_chain_nt<4>(a, num_sms, s);
  if (a.N <= 8) return launch_chain_nt<8>(a, num_sms, s);
  return launch_chain_nt<16>(a, num_sms, s);
}

}  // namespace ge
