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
// Work split: one block per SM with CW consumer warps (16 for up to four
// tokens, the weight rows then cut in two segments; 8 with whole rows
// otherwise) and P producer warps. Block b owns rows [b*M/G, (b+1)*M/G) of
// every layer (G blocks); its items (row segments, layer after layer) pass
// through one ring of S segment-sized slots in shared memory, item i in slot
// i % S: producer warp g (one lane) issues items g, g + P, ... as 1-D bulk
// copies counted on the slot's "full" mbarrier, once the consumer of the
// slot's previous item has arrived on its "empty" mbarrier and once no more
// than F of its own copies are in flight; consumer warp w takes rows w,
// w + CW, ... of every layer. When the ring is shorter than a layer, a
// per-slot tag (the item last issued into it) tells a consumer that its item
// is the one in the slot.
//
// Layer boundary: every block stages the N x K activations of layer l in
// shared memory from the exchange words the blocks wrote for layer l - 1:
// 32-bit words, the 16-bit output in the low half and a (launch, layer) tag
// in the high half, double-buffered by layer parity. A block's thread waits
// for a relaxed per-layer arrival count to reach G (every block has issued
// its stores), then every thread waits on its own words until they carry the
// tag: the data is its own flag, so no fence orders the stores before the
// count and the count's add never waits for them. Then, per item: wait for
// the slot, fp32 dot products from shared memory (the 16-bit products
// widened exactly), release the slot; after a row's last segment, butterfly
// reduction, bias + activation, round, store to Y and to the exchange.
// Every wait is bounded: an expired wait sets ERR_CHAIN_TIMEOUT and a
// grid-wide abort flag, the abort decision is taken at a barrier in every
// consumer thread at once, and every producer waits (bounded) for its
// copies in flight before the block exits. The last block to finish clears
// the counts and the flag and advances the launch epoch.
//
// Measured on 32 layers of 4096 x 4096 fp16, one token (one launch, L2
// flushed, all variants on one GPU): 8.2 us a layer with every warp issuing
// its own rows into a ring of its own and a release/acquire count per
// layer; 7.6-7.7 with the producer warps and that count; 6.7-6.8 with the
// tagged exchange (4.95 TB/s). Stamps of that count form showed the release
// add waiting ~1 us for the block's stores and the acquire poll plus the
// activation load two more L2 round trips. One producer thread issues a copy
// only every ~400 SM cycles (its mbarrier probes and the copy are
// latency-bound): one producer gave 16.9 us a layer, three 7.2; 27 lanes of
// one warp as producers were slower (8.8), so were whole-row items (7.6),
// requesting the next layers into L2 ahead of the ring (+11-25 %) or just
// the items whose slots are still busy (+21 %), pacing the issue, and
// polling the exchange words without the count (8.5-9 us a layer even with
// a back-off between polls), and several copies of the exchange for the
// readers to spread over (2-16 copies: 6.9-7.9 us, the extra stores cost); four or six producer warps were slower than three (7.25,
// 7.41: their waits take issue slots from the consumer warps). Capping the
// copies in flight at half the ring gained a little over none (6.77
// against 7.00), and any cap from 12 to 30 measures the same (213.6-215.7
// us). Without the wait for the previous layer's outputs (a
// scratch copy computing on stale activations) the same ring streams at
// 5.84 us a layer (5.46 with no cap on the copies in flight): the layer
// boundary costs ~0.9 us a layer. Two ways of hiding it were slower:
// issuing all of a thread's exchange-word loads before checking the first
// (215.7 us either way: the wait is for the last block's words, not for
// round trips), and a half-split order -- each block's rows in a first-half
// and a second-half part, segment-major, each half of the outputs counted
// and staged on its own so that the first half's exchange could overlap
// the second half's work -- 230-232 us against 215: the ring has already
// fetched the next layer, so the consumers reach each half's wait almost
// at once, and the two extra barriers a layer hold every warp to the
// slowest. L2 prefetches issued while a block waits at the boundary were
// slower still (the next layer's first 18 segments: 277 us; the current
// layer's last 27: 249 us). Stamps of the tagged form, per layer: ~0.5 us until the
// count shows every block's stores issued, ~1.2 us until every word of the
// previous layer has arrived and is staged, ~3.5 us until the last weight
// segment of the layer has landed (a quarter of them are issued after the
// staging), ~0.8 us for the last rows' dot products and stores.
#include <atomic>

#include "ge_internal.h"
#include "ge_ptx.cuh"

namespace ge {
namespace {

constexpr int kSmemMax = 232448;        // dynamic shared memory per block
constexpr int kSmemSlack = 128 + 16;    // base alignment + the block's flags
constexpr int kMaxProducers = 3;

__device__ __forceinline__ float chain_act(int epi, float z) {
  if (epi == EPI_RELU_BIAS) return fmaxf(z, 0.0f);
  if (epi == EPI_GELU_BIAS) return gelu_tanh(z);
  if (epi == EPI_GELU_ERF_BIAS) return gelu_erf(z);
  return z;
}

// Named barrier 1 over the consumer warps (the producer warps never join
// it); the _or form returns, in every thread, whether any thread passed
// `pred` -- one decision for all of them, whatever a flag reads later.
__device__ __forceinline__ void consumers_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}
__device__ __forceinline__ bool consumers_sync_or(int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n"
      ".reg .pred p, q;\n"
      "setp.ne.u32 p, %1, 0;\n"
      "bar.red.or.pred q, 1, %2, p;\n"
      "selp.u32 %0, 1, 0, q;\n"
      "}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(nthreads)
      : "memory");
  return r != 0;
}

size_t x_bytes(int K, int N) { return (static_cast<size_t>(N) * K * 2 + 127) & ~static_cast<size_t>(127); }

// Launch shape: consumer warps per block and segments per weight row (one
// ring item is one segment). Wide rows of few tokens take 16 warps and
// half-row items: twice the rows in progress at once.
struct Shape {
  int warps, seg;
};
Shape chain_shape(int K, int N) {
  if (N <= 4 && K % 16 == 0) return {16, 2};
  return {8, 1};
}

// Ring slots per block beside the staged activations (each a segment, its
// two mbarriers and its item tag).
constexpr int kSlotExtra = 8 + 8 + 4;
int slots_for(int K, int N, Shape sh) {
  const long long seg_bytes = 2LL * K / sh.seg;
  const long long avail = kSmemMax - kSmemSlack - static_cast<long long>(x_bytes(K, N));
  long long r = avail > 0 ? avail / (seg_bytes + kSlotExtra) : 0;
  if (r > 4096) r = 4096;
  return static_cast<int>(r);
}

size_t chain_smem(int K, int N, Shape sh, int slots) {
  return kSmemSlack + x_bytes(K, N) + static_cast<size_t>(slots) * (2ull * K / sh.seg + kSlotExtra);
}

// CW consumer warps and p.producers (1..kMaxProducers) producer warps per block.
template <int NT, bool BF16, int CW, int SEG>
__global__ void __launch_bounds__(32 * (CW + kMaxProducers), 1) gemv_chain_kernel(const __grid_constant__ ChainArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t row_bytes = static_cast<uint32_t>(p.K) * 2u;
  const uint32_t seg_bytes = row_bytes / SEG;
  const int C16 = (p.K >> 3) / SEG;  // 16-byte chunks per segment
  const int S = p.slots;
  const size_t xb = (static_cast<size_t>(p.N) * row_bytes + 127) & ~static_cast<size_t>(127);
  uint8_t* xs = smem;
  uint8_t* ring = smem + xb;
  const uint32_t ring_s = smem_u32(ring);
  uint8_t* bars = ring + static_cast<size_t>(S) * seg_bytes;
  const uint32_t full0 = smem_u32(bars);           // slot s landed: full0 + 8 s
  const uint32_t empty0 = full0 + 8u * S;          // slot s consumed: empty0 + 8 s
  volatile int* tags = reinterpret_cast<volatile int*>(bars + 16 * S);  // the last item issued into slot s
  volatile int* abort_s = tags + S;
  volatile int* never = abort_s + 1;
  unsigned int* const epoch_g = p.sync;  // advanced by the last block of every launch
  unsigned int* const done = p.sync + 1;
  volatile unsigned int* const abort_g = p.sync + 2;
  unsigned int* const arrived = p.sync + 3;  // blocks that stored layer l: arrived[l]

  const int r0 = static_cast<int>(static_cast<long long>(blockIdx.x) * p.M / gridDim.x);
  const int r1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * p.M / gridDim.x);
  const int PL = (r1 - r0) * SEG;                              // the block's items per layer
  const int total = PL * p.layers;  // the block's items (the launcher bounds it)

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, 1);
      tags[s] = -1;
    }
    *abort_s = 0;
    *never = 0;
  }
  fence_barrier_init();
  __syncthreads();

  if (warp >= CW) {
    // Producers: the block's items in order -- layer l, row r0 + j, segment
    // h is item l * PL + j * SEG + h, in slot (item % S) -- producer warp g
    // (lane 0) issuing items g, g + P, ..., each once its slot's previous
    // item is consumed. P divides S, so slot s only ever holds producer
    // (s % P)'s items: the producer itself issued the slot's previous item
    // after that item's predecessor was consumed, and the slot's barriers are
    // never more than one phase from the parity it waits for. Slots, phases,
    // layers and rows advance by counting (no divisions).
    const int P = p.producers;
    const int g = warp - CW;
    if (lane == 0 && GE_DCHECK(S % P == 0, p.err)) {
      int i = g;
      int s = g % S, ph = (g / S) & 1;  // slot and phase of item i
      const int F = p.inflight;                 // a multiple of P, at most S
      int su = g - F, phu = 0;                  // slot and phase of item i - F
      while (su < 0) {
        su += S;
        phu ^= 1;
      }
      int l = 0, q = g;       // item i's layer and index in it
      while (PL > 0 && q >= PL) {
        q -= PL;
        ++l;
      }
      const uint8_t* al = l < p.layers ? reinterpret_cast<const uint8_t*>(p.A[l]) : nullptr;
      for (; i < total; i += P) {
        if (i >= S && !mbar_wait_bounded(empty0 + 8u * s, static_cast<uint32_t>(ph ^ 1), abort_s, p.budget)) {
          if (!*abort_s) {
            atomicOr(p.err, ERR_CHAIN_TIMEOUT);
            *abort_g = 1;
            *abort_s = 1;
          }
          break;
        }
        // at most F copies in flight: item i - F (this producer's own, F a
        // multiple of P) has landed
        // (GE_DEBUG) su is item i - F's slot
        const bool capped = i >= F && F < S && GE_DCHECK(su == (i - F) % S, p.err);
        const bool ok = !capped || mbar_wait_bounded(full0 + 8u * su, static_cast<uint32_t>(phu), abort_s, p.budget);
        for (su += P; su >= S; su -= S) phu ^= 1;  // item i - F advances with i, waited for or not
        if (!ok) {
          if (!*abort_s) {
            atomicOr(p.err, ERR_CHAIN_TIMEOUT);
            *abort_g = 1;
            *abort_s = 1;
          }
          break;
        }
        const long long row = r0 + q / SEG;
        // (GE_DEBUG) the item's layer, row and slot lie in range; a skipped
        // copy ends in the consumer's bounded wait
        if (!GE_DCHECK(l < p.layers && row < r1 && s == i % S, p.err)) break;
        tags[s] = i;
        mbar_arrive_expect_tx(full0 + 8u * s, seg_bytes);
        bulk_load_1d(ring_s + static_cast<uint32_t>(s) * seg_bytes, al + row * p.lda * 2 + (q % SEG) * seg_bytes,
                     seg_bytes, full0 + 8u * s);
        for (s += P; s >= S; s -= S) ph ^= 1;
        q += P;
        if (q >= PL) {
          while (q >= PL) {
            q -= PL;
            ++l;
          }
          if (l < p.layers) al = reinterpret_cast<const uint8_t*>(p.A[l]);
        }
      }
      // This producer's copies still in flight must land before the block's
      // shared memory goes away (after an abort some were never waited for).
      for (int u = i - P; u >= 0 && u >= i - S; u -= P)
        if (!mbar_wait_bounded(full0 + 8u * static_cast<uint32_t>(u % S), static_cast<uint32_t>((u / S) & 1), never,
                               p.budget))
          atomicOr(p.err, ERR_DRAIN_TIMEOUT);
    }
  } else {
    // Consumers: warp w takes rows j = w, w + CW, ... of every layer.
    const int nthreads = 32 * CW;
    // Layer l's outputs reach the other blocks as exchange words tagged
    // etag | l, etag naming this launch (never 0, and different from the
    // previous launch's); each launch writes both halves of the exchange, so
    // no word from an earlier launch carries a tag this one waits for.
    const unsigned int etag = ((*reinterpret_cast<volatile unsigned int*>(epoch_g) % 1023u) + 1u) << 6;
    const long long MN = static_cast<long long>(p.N) * p.M;
    for (int l = 0; l < p.layers; ++l) {
      // The bias of this warp's rows of the layer, requested before the wait
      // for the previous layer: lane k holds row (warp + CW k)'s (the first
      // 32 rows); kept as loaded and converted at use.
      const unsigned short* bias = p.bias[l];
      const int nrw = r1 - r0 > warp ? (r1 - r0 - warp + CW - 1) / CW : 0;
      unsigned short braw = 0;
      if (p.epi != EPI_NONE && lane < nrw) braw = bias[r0 + warp + CW * lane];
      // this layer's activations into shared memory: X, or the previous
      // layer's outputs as every block writes them -- once the relaxed count
      // says every block has issued its stores, each exchange word is waited
      // for until it carries the previous layer's tag (the data is its own
      // flag: no fence orders the stores before the count)
      if (l == 0) {
        const int K16 = p.K >> 3;
        for (int e = threadIdx.x; e < p.N * K16; e += nthreads) {
          const int n = e / K16;
          const int c = e - n * K16;
          *reinterpret_cast<uint4*>(xs + static_cast<size_t>(n) * row_bytes + 16 * c) = ld_cg_u4(p.X + n * p.ldx + 8 * c);
        }
        consumers_sync(nthreads);
      } else {
        // every block has issued its stores of layer l - 1 (a relaxed count:
        // the words themselves say when they have arrived)
        if (threadIdx.x == 0) {
          const long long t0 = clock64();
          while (ld_relaxed_gpu_u32(arrived + (l - 1)) < gridDim.x) {
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
        if (consumers_sync_or(nthreads, *abort_s != 0)) break;
        const uint32_t want = (etag | static_cast<uint32_t>(l - 1)) << 16;
        const unsigned int* xb = p.xbuf + ((l - 1) & 1) * MN;
        const int K4 = p.K >> 2;
        bool ok = true;
        for (int e = threadIdx.x; e < p.N * K4 && ok; e += nthreads) {
          const int n = e / K4;
          const int c = e - n * K4;
          const unsigned int* src = xb + static_cast<long long>(n) * p.M + 4 * c;
          uint4 v = ld_relaxed_gpu_u4(src);
          if (((v.x & v.y & v.z & v.w) >> 16) != (want >> 16) || ((v.x | v.y | v.z | v.w) >> 16) != (want >> 16)) {
            const long long t0 = clock64();
            while (true) {
              v = ld_relaxed_gpu_u4(src);
              if (((v.x & v.y & v.z & v.w) >> 16) == (want >> 16) && ((v.x | v.y | v.z | v.w) >> 16) == (want >> 16))
                break;
              if (*abort_g != 0 || *abort_s != 0) {
                *abort_s = 1;
                ok = false;
                break;
              }
              if (clock64() - t0 > p.budget) {
                atomicOr(p.err, ERR_CHAIN_TIMEOUT);
                *abort_g = 1;
                *abort_s = 1;
                ok = false;
                break;
              }
            }
          }
          *reinterpret_cast<uint2*>(xs + static_cast<size_t>(n) * row_bytes + 8 * c) =
              make_uint2((v.x & 0xFFFFu) | (v.y << 16), (v.z & 0xFFFFu) | (v.w << 16));
        }
        if (consumers_sync_or(nthreads, !ok || *abort_s != 0)) break;
      }
      unsigned short* ydst = p.Y + static_cast<long long>(l) * p.N * p.ldy;
      // two accumulators per token (alternate 16-byte chunks) halve the chain
      // of dependent multiply-adds; added in a fixed order at the row's end
      float acc[NT], acc2[NT];
      bool failed = false;
      for (int k = 0; k < nrw && !failed; ++k) {
        const int j = warp + CW * k;
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[n] = acc2[n] = 0.0f;
        for (int h = 0; h < SEG; ++h) {
          const int it = l * PL + j * SEG + h;
          const int s = it % S;
          // The slot's tag names the item last issued into it. Other warps'
          // items share the slot when the ring is shorter than a layer, and
          // its barrier's parity alone cannot tell this item's phase from
          // one two phases earlier: wait for the tag first.
          bool tagged = true;
          if (S < PL && tags[s] != it) {
            const long long t0 = clock64();
            while (tags[s] != it)
              if (*abort_s || clock64() - t0 > p.budget) {
                tagged = false;
                break;
              }
          }
          const bool landed =
              tagged && mbar_wait_bounded(full0 + 8u * s, static_cast<uint32_t>((it / S) & 1), abort_s, p.budget);
          if (!__all_sync(0xffffffffu, landed)) {
            if (lane == 0 && !*abort_s) {
              atomicOr(p.err, ERR_CHAIN_TIMEOUT);
              *abort_g = 1;
              *abort_s = 1;
            }
            failed = true;
            break;
          }
          const uint8_t* wseg = ring + static_cast<size_t>(s) * seg_bytes;
          const uint8_t* xseg = xs + static_cast<size_t>(h) * seg_bytes;
          int c = lane;
          for (; c + 32 < C16; c += 64) {
            const uint4 w0 = *reinterpret_cast<const uint4*>(wseg + 16 * c);
            const uint4 w1 = *reinterpret_cast<const uint4*>(wseg + 16 * (c + 32));
#pragma unroll
            for (int n = 0; n < NT; ++n)
              if (n < p.N) {
                const uint8_t* xr = xseg + static_cast<size_t>(n) * row_bytes;
                acc[n] = dot8_mixed<BF16>(w0, *reinterpret_cast<const uint4*>(xr + 16 * c), acc[n]);
                acc2[n] = dot8_mixed<BF16>(w1, *reinterpret_cast<const uint4*>(xr + 16 * (c + 32)), acc2[n]);
              }
          }
          if (c < C16) {
            const uint4 w0 = *reinterpret_cast<const uint4*>(wseg + 16 * c);
#pragma unroll
            for (int n = 0; n < NT; ++n)
              if (n < p.N)
                acc[n] = dot8_mixed<BF16>(
                    w0, *reinterpret_cast<const uint4*>(xseg + static_cast<size_t>(n) * row_bytes + 16 * c), acc[n]);
          }
          // the slot is consumed: the producer may refill it (these
          // shared-memory reads are ordered before the bulk copy's writes)
          __syncwarp();
          if (lane == 0) {
            fence_proxy_async_smem();
            mbar_arrive(empty0 + 8u * s);
          }
        }
        if (failed) break;
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
        const unsigned short bj = k < 32 ? static_cast<unsigned short>(__shfl_sync(0xffffffffu, braw, k)) : 0;
        if (lane < p.N) {
          const long long row = r0 + j;
          if (p.epi != EPI_NONE) z += to_f32(BF16, k < 32 ? bj : bias[row]);
          const unsigned short y = from_f32(BF16, chain_act(p.epi, z));
          ydst[static_cast<long long>(lane) * p.ldy + row] = y;
          const uint32_t word = ((etag | static_cast<uint32_t>(l)) << 16) | y;
          unsigned int* xw = p.xbuf + (l & 1) * MN + static_cast<long long>(lane) * p.M + row;
          st_relaxed_gpu_u32(xw, word);
          if (p.layers == 1) st_relaxed_gpu_u32(xw + MN, word);  // both halves, every launch
        }
      }
      // every warp is done with this layer's activations before the next
      // layer's replace them, and has issued its stores of the layer
      if (consumers_sync_or(nthreads, failed || *abort_s != 0)) break;
      if (threadIdx.x == 0) red_relaxed_gpu_add(arrived + l, 1u);
    }
  }
  __syncthreads();
  // The last block to get here is past every wait of every block: it
  // advances the launch epoch and clears the abort flag for the next launch.
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned int prev = atomicAdd(done, 1u);
    if (prev == gridDim.x - 1) {
      *epoch_g = *epoch_g + 1u;
      for (int l = 0; l < p.layers; ++l) arrived[l] = 0u;
      *abort_g = 0u;
      __threadfence();
      atomicExch(done, 0u);
    }
  }
}

template <int NT, bool BF16, int CW, int SEG>
cudaError_t launch_chain_t(const ChainArgs& args, int num_sms, cudaStream_t s) {
  static std::atomic<bool> configured[64] = {};
  ChainArgs a = args;
  const Shape sh{CW, SEG};
  a.slots = slots_for(a.K, a.N, sh);
  if (a.slots < 1) return cudaErrorInvalidValue;
  // item indices are 32-bit: rows per block x segments x layers
  if ((static_cast<long long>(a.M) / num_sms + 1) * SEG * a.layers >= (1LL << 30)) return cudaErrorInvalidValue;
  // Producer warps issuing the bulk copies (args.producers if the caller
  // asks for 1..kMaxProducers), and the ring's slots cut to a multiple of
  // their number (each slot then belongs to one producer).
  a.producers = args.producers >= 1 && args.producers <= kMaxProducers ? args.producers : kMaxProducers;
  if (a.producers > a.slots) a.producers = a.slots;
  a.slots -= a.slots % a.producers;
  // Copies in flight per block (args.inflight if asked; a multiple of the
  // producers, at most the slots): enough to keep the block's share of HBM
  // busy, few enough that a copy issued at a layer boundary does not queue
  // behind a deep backlog of other blocks' copies. Default half the ring.
  a.inflight = args.inflight >= 1 ? args.inflight : a.slots / 2;
  if (a.inflight < 1) a.inflight = 1;
  a.inflight = (a.inflight + a.producers - 1) / a.producers * a.producers;
  if (a.inflight > a.slots) a.inflight = a.slots;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(gemv_chain_kernel<NT, BF16, CW, SEG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemMax);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  const size_t smem = chain_smem(a.K, a.N, sh, a.slots);
  const int threads = 32 * (CW + a.producers);
  // The blocks wait on one another: all of them must be resident at once,
  // which the cooperative launch guarantees (or refuses).
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_chain_kernel<NT, BF16, CW, SEG>, threads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms), 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
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

int gemv_chain_slots(int K, int N) { return slots_for(K, N, chain_shape(K, N)); }

cudaError_t launch_gemv_chain(const ChainArgs& a, int num_sms, cudaStream_t s) {
  if (a.N <= 1) return launch_chain_nt<1>(a, num_sms, s);
  if (a.N <= 2) return launch_chain_nt<2>(a, num_sms, s);
  if (a.N <= 4) return launch_chain_nt<4>(a, num_sms, s);
  if (a.N <= 8) return launch_chain_nt<8>(a, num_sms, s);
  return launch_chain_nt<16>(a, num_sms, s);
}

}  // namespace ge
