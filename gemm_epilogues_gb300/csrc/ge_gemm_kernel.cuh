// ge_gemm_kernel.cuh -- persistent, warp-specialised tcgen05 GEMM with the
// fused bias + activation (+ ReLU mask) epilogue, for sm_103a. Included by
// one translation unit per epilogue code (ge_gemm_epi_*.cu), each of which
// instantiates launch_tc_gemm_epi<EPI> for every tile shape: with the
// epilogue a compile-time constant, a kernel's per-slab loop holds only its
// own epilogue's instructions (measured on an epilogue-bound problem, 8192 x
// 8192 x 128 with no bias: 9.3 -> 4.5 us per 256 x 256 tile with the slab
// loop reduced to one epilogue; the loop of every epilogue together did not
// stay in the instruction cache).
//
// What it computes (page title, section):
//  * nvmath-python cuBLASLt bias-fusion guide, "Core API and parameter
//    configuration" and "Principle of the performance gain": the product and
//    the bias add happen in one kernel and the result is written to global
//    memory once, the bias (m,1) broadcast over the columns.
//  * same page, "Advanced techniques": ReLU / GELU fused after the bias;
//    fp16 operands, 32-bit accumulation, fp16 output.
//  * Fusing bias addition with matrix multiplication using nvmath-python:
//    the intermediate WX never goes back to global memory; RELU_AUX_BIAS
//    also keeps the auxiliary output the backward pass needs.
//
// Structure (one CTA per SM, 96 + 32 * EPIW threads; 192 + 32 * EPIW with AM):
//   warp 0      TMA producer: A and B k-slices (64 fp16 = one 128-byte
//               swizzle row) into a STAGES-deep shared-memory ring.
//   warp 1      owns TMEM (2 x BN fp32 columns: a double-buffered 128 x BN
//               accumulator) and one lane issues tcgen05.mma 128 x BN x 16.
//   warps 2..   EPIW = 4 or 8 epilogue warps: tcgen05.ld a 32-row x
//               32-column slab of the accumulator, add the bias, apply the
//               activation, build the mask word, round to fp16, stage in
//               64-byte-swizzled shared memory and TMA-store it; runs while
//               the MMA warp already accumulates the next tile into the
//               other TMEM buffer. With 8, two warps share each TMEM lane
//               quarter (warp % 4) and take alternate slabs, so the heaviest
//               epilogue (the GELU derivative) keeps pace with the MMAs.
//   (AM)        four more warps clear the masked elements of each stage's A
//               tile in shared memory before the MMA reads it (the weight
//               gradient with the ReLU backward on its operand).
//   (else)      one more warp: a second producer that issues the B loads
//               when asked (p.two_producers: an M/N-major operand makes a
//               stage three or four boxes, and one thread issues a box only
//               every few hundred cycles); otherwise it idles.
// Pair mode (PAIR = true, clusters of 2 CTAs on 2 SMs): the tile is 256 x BN;
// each CTA stages its own 128 rows of A and its own half of B's BN columns,
// the even CTA issues tcgen05.mma.cta_group::2 (M = 256) which reads both
// CTAs' shared memory and writes both CTAs' TMEM, and every commit is
// multicast to both CTAs. Per SM this moves a third less shared-memory
// traffic per flop than the single-CTA 128 x BN tile.
// Every wait is bounded; an expired wait records a bit in the error word,
// raises a CTA-wide abort flag, and every role drains its in-flight copies
// before the CTA frees TMEM and exits.
#pragma once

#include <atomic>

#include "ge_internal.h"
#include "ge_ptx.cuh"

namespace ge {
namespace {

constexpr int BM = 128;            // accumulator rows = TMEM lanes
constexpr int BK = 64;             // 16-bit k-values in one 128-byte swizzle row (one panel)

constexpr int EPI_BUF_BYTES = 32 * 64;  // 32 rows x 32 fp16 columns

// EPIW = epilogue warps: 4 (one per TMEM lane quarter) or 8 (two per quarter,
// taking alternate 32-column slabs). AM = the A operand is masked in shared
// memory by four more warps before the MMA reads it (DW_DRELU_BGRAD).
// KB = k-values per stage: 64 (one panel) or 128 (two panels, each operand
// fetched in one box of up to 32 KB: the TMA unit moves large boxes at a
// higher rate than several small ones).
template <int BN, bool PAIR, int EPIW, bool AM = false, int KB = 64>
struct Cfg {
  static constexpr int EPI_WARPS = EPIW;
  static constexpr int XFORM_WARPS = AM ? 4 : 0;
  // (+1 warp without AM: the second producer, issuing B, when asked)
  static constexpr int NUM_THREADS = 64 + 32 * EPIW + 32 * XFORM_WARPS + (AM ? 0 : 32);
  static constexpr int HALVES = EPIW / 4;  // warps per lane quarter
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // B columns staged by one CTA
  static_assert(KB == 64 || (KB == 128 && !AM), "k-values per stage");
  static constexpr int PANELS = KB / BK;
  static constexpr int A_BYTES = BM * KB * 2;
  static constexpr int B_BYTES = B_ROWS * KB * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (196608 / STAGE_BYTES) < 8 ? (196608 / STAGE_BYTES) : 8;
  static constexpr int OFF_EPI = STAGES * STAGE_BYTES;
  static constexpr int EPI_BYTES = EPI_WARPS * 2 * EPI_BUF_BYTES;
  // AM: per stage, the mask words of the stage's BK k-rows for this CTA's
  // BM rows of A' (BK x BM/32 words = 1 KB), loaded with the operands.
  static constexpr int MASK_SLOT = BK * (BM / 32) * 4;
  static constexpr int OFF_MASK = OFF_EPI + EPI_BYTES;
  static constexpr int MASK_BYTES = AM ? STAGES * MASK_SLOT : 0;
  static constexpr int OFF_BAR = OFF_MASK + MASK_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 5 + (AM ? STAGES : 0);
  static constexpr int OFF_MISC = OFF_BAR + 8 * NUM_BARS;
  // misc: TMEM address, abort flag, a flag that is never set, then (GE_DEBUG)
  // the producer's fill count of each stage
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 4 * 8 + 1024;  // + 1 KB for base alignment
  static constexpr int TMEM_COLS = 2 * BN;  // columns in use (two accumulators)
  // the allocation: a power of two of at least 32 columns
  static constexpr int TMEM_ALLOC = TMEM_COLS <= 32 ? 32 : TMEM_COLS <= 64 ? 64 : TMEM_COLS <= 128 ? 128
                                  : TMEM_COLS <= 256 ? 256 : 512;
  static_assert(TMEM_COLS <= 512 && B_ROWS % 8 == 0, "tile width");
  static constexpr int TILE_M = PAIR ? 2 * BM : BM;
  static constexpr int EPI_ARRIVALS = PAIR ? 2 * EPI_WARPS : EPI_WARPS;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(STAGE_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "SW128 atoms need 1 KB alignment");
};

__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int group_m, int& mt,
                                            int& nt) {
  const int per_group = group_m * num_n;
  const int g = tile / per_group;
  const int first_m = g * group_m;
  const int gsz = min(num_m - first_m, group_m);
  const int r = tile - g * per_group;
  mt = first_m + r % gsz;
  nt = r / gsz;
}

// Work unit u -> tile and k-block range. Units below tail_start are whole
// tiles; the rest are `split` consecutive k-ranges of each tail tile.
// v >= 0 is the unit's index into the partial-sum workspace.
__device__ __forceinline__ void unit_info(int u, int tail_start, int split, int num_kb, int& tile,
                                          int& kb0, int& kb1, int& v) {
  if (u < tail_start) {
    tile = u;
    kb0 = 0;
    kb1 = num_kb;
    v = -1;
  } else {
    v = u - tail_start;
    tile = tail_start + v / split;
    const int s = v % split;
    kb0 = s * num_kb / split;
    kb1 = (s + 1) * num_kb / split;
  }
}

// Stream-K: worker w's share of the I iterations starts at w * I / W.
__device__ __forceinline__ long long sk_begin(long long w, long long iters, long long workers) {
  return w * iters / workers;
}

// Unit kinds besides v >= 0 (an fp32 piece for slot / piece v): a whole tile
// with its epilogue, and the stream-K segment that starts a tile and
// finishes it with the pieces of the workers that hold the tile's rest.
constexpr int kWhole = -1;
constexpr int kFinish = -2;

// The work of one worker, in the same order for every role of the CTA: its
// data-parallel units u = worker, worker + W, ... (whole tiles below
// tail_start, split-K pieces of the tiles above), then its stream-K
// iterations [it, it_end) of the last sk_tiles tiles, cut at tile
// boundaries. Only the first stream-K segment can start inside a tile
// (it is spilled to slot `worker`) and only the last can start a tile
// without ending it (it finishes that tile).
struct Sched {
  int u, step, num_units, tail_start, split, num_kb, dp_tiles, worker;
  long long it, it_end;
  __device__ __forceinline__ bool next(int& tile, int& kb0, int& kb1, int& v, int& u_dp) {
    if (u < num_units) {
      unit_info(u, tail_start, split, num_kb, tile, kb0, kb1, v);
      u_dp = u;
      u += step;
      return true;
    }
    if (it < it_end) {
      const long long t = it / num_kb;
      kb0 = static_cast<int>(it - t * num_kb);
      const long long left = it_end - it;
      kb1 = left < num_kb - kb0 ? kb0 + static_cast<int>(left) : num_kb;
      tile = dp_tiles + static_cast<int>(t);
      v = (kb0 == 0 && kb1 == num_kb) ? kWhole : (kb0 > 0 ? worker : kFinish);
      u_dp = -1;
      it += kb1 - kb0;
      return true;
    }
    return false;
  }
};

__device__ __forceinline__ float apply_act(int epi, float z) {
  if (epi == EPI_RELU_BIAS || epi == EPI_RELU_AUX_BIAS) return fmaxf(z, 0.0f);
  if (epi == EPI_GELU_BIAS || epi == EPI_GELU_AUX_BIAS) return gelu_tanh(z);
  if (epi == EPI_GELU_ERF_BIAS) return gelu_erf(z);
  return z;
}

// Epilogue of one 32-column slab held by this thread (one accumulator row;
// bcol[j] is the bias of its column j, the row's bias repeated when the bias
// is per row). Returns the 32 packed 16-bit values in `packed`, the mask
// bits, and for GELU_AUX_BIAS the packed pre-activations in `zpacked`.
template <int EPI>
__device__ __forceinline__ uint32_t epilogue_slab(const uint32_t (&v)[32], const float (&bcol)[32],
                                                  uint32_t (&packed)[16], uint32_t (&zpacked)[16], bool bf16) {
  uint32_t bits = 0;
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    float z0 = __uint_as_float(v[j]);
    float z1 = __uint_as_float(v[j + 1]);
    if (EPI != EPI_NONE) {
      z0 += bcol[j];
      z1 += bcol[j + 1];
    }
    if (EPI == EPI_RELU_AUX_BIAS) {
      bits |= (z0 > 0.0f ? 1u : 0u) << j;
      bits |= (z1 > 0.0f ? 1u : 0u) << (j + 1);
    }
    if (EPI == EPI_GELU_AUX_BIAS) zpacked[j / 2] = pack2(bf16, z0, z1);
    packed[j / 2] = pack2(bf16, apply_act(EPI, z0), apply_act(EPI, z1));
  }
  return bits;
}

// This thread's 32 16-bit values of a row-major input laid out like D'
// (DGELU_BGRAD's z, BIAS_RESIDUAL's residual) at row grow, columns gcol0..,
// packed in pairs; 0 past the matrix.
__device__ __forceinline__ void load_slab16(const GemmArgs& p, int grow, int gcol0, uint32_t (&zw)[16]) {
  const unsigned short* zrow = p.zaux + static_cast<long long>(grow) * p.ld_zaux + gcol0;
  if (grow < p.Mk && gcol0 + 32 <= p.Nk) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(zrow) + i);
      zw[4 * i] = w.x;
      zw[4 * i + 1] = w.y;
      zw[4 * i + 2] = w.z;
      zw[4 * i + 3] = w.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t lo = grow < p.Mk && gcol0 + 2 * j < p.Nk ? zrow[2 * j] : 0u;
      const uint32_t hi = grow < p.Mk && gcol0 + 2 * j + 1 < p.Nk ? zrow[2 * j + 1] : 0u;
      zw[j] = lo | (hi << 16);
    }
  }
}

// One 32x32 slab of 16-bit values (row `grow` of this thread; the warp's 32
// rows start at `rbase`) to global memory at columns gcol0.. of a row-major
// matrix `dst` (ld elements per row, tensor map `map`). A slab whose end
// runs past Nk at a column that is not on a 16-byte boundary is stored
// element by element (a TMA store writes whole 16-byte chunks and would
// spill into the caller's columns). Otherwise the slab is staged in shared
// memory (64-byte swizzle: 16-byte chunk j of row r sits at chunk
// j ^ ((r >> 1) & 3)) and TMA-stored; the two staging buffers alternate per
// issued store, so the newest store in flight always reads the other buffer. `dry` (the epilogue's instruction-cache warm-up, before
// any store of the CTA is in flight) stages the slab and stores nothing.
__device__ __forceinline__ void store_slab(const uint32_t (&packed)[16], const CUtensorMap* map,
                                           unsigned short* dst, long long ld, int gcol0, int rbase,
                                           int grow, int Mk, int Nk, uint8_t* stg, int& nstore,
                                           int lane, unsigned int* dbg_err, bool dry) {
  (void)dbg_err;
  if (gcol0 + 32 > Nk && (Nk & 7) != 0) {
    if (grow < Mk && !dry) {
      unsigned short* drow = dst + static_cast<long long>(grow) * ld + gcol0;
      const int nvalid = Nk - gcol0;
#pragma unroll
      for (int j = 0; j < 32; ++j) {  // static indices keep packed[] in registers
        if (j < nvalid) {
          const uint32_t w = packed[j >> 1];
          drow[j] = static_cast<unsigned short>((j & 1) ? (w >> 16) : (w & 0xFFFFu));
        }
      }
    }
  } else if (rbase < Mk) {
    uint8_t* buf = stg + (nstore & 1) * EPI_BUF_BYTES;
#ifdef GE_DEBUG
    if (lane == 0 && (gcol0 < 0 || gcol0 % 8 != 0 || rbase < 0)) atomicOr(dbg_err, ERR_DEBUG_CHECK);
#endif
    if (lane == 0 && nstore >= 2 && !dry) bulk_wait_group_read<1>();
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int sw = j ^ ((lane >> 1) & 3);
      *reinterpret_cast<uint4*>(buf + lane * 64 + sw * 16) =
          make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (dry) return;
    if (lane == 0) {
      tma_store_2d(map, smem_u32(buf), gcol0, rbase);
      bulk_commit_group();
    }
    ++nstore;
  }
}

template <int EPI, int BN, bool PAIR, int EPIW, bool AM = false, int KB = 64>
__global__ void __launch_bounds__(64 + 32 * EPIW + (AM ? 128 : 32), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmZ,
                   const GemmArgs p) {
  using C = Cfg<BN, PAIR, EPIW, AM, KB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * C::STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * C::STAGES + 4);
  // AM: stage s of A' has been masked (the MMA waits on this instead of the
  // load's barrier); counted on the pair's leader for both CTAs' warps.
  auto xform_bar = [&](int s) { return bar0 + 8u * (2 * C::STAGES + 5 + s); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* never = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  // GE_DEBUG: fills issued into each stage (the MMA warp checks that the
  // producer is never more than one phase of a stage ahead of it)
  volatile unsigned int* dbg_fills = reinterpret_cast<volatile unsigned int*>(smem + C::OFF_MISC + 16);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;  // CTA within the cluster
  const uint32_t pr = rank & 1u;                         // CTA within its pair
  const uint32_t lead = rank & ~1u;                      // the pair's MMA-issuing CTA
  const bool leader = pr == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), C::EPI_ARRIVALS);
    }
    mbar_init(drain_bar, 1);
    if constexpr (AM)
      for (int s = 0; s < C::STAGES; ++s) mbar_init(xform_bar(s), (PAIR ? 2 : 1) * C::XFORM_WARPS);
    *abort_flag = 0;
    *never = 0;
    for (int s = 0; s < C::STAGES && s < 8; ++s) dbg_fills[s] = 0u;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmD);
    if (EPI == EPI_GELU_AUX_BIAS || AM) tma_prefetch_desc(&tmZ);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_ALLOC);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), C::TMEM_ALLOC);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync();  // the peer's barriers exist before anything targets them
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // A dependent launched with programmatic serialization (the split-K fixup,
  // a decode GEMV) may be scheduled from here on; it waits in the kernel
  // for this grid to complete before it reads what this grid writes.
  grid_launch_dependents();

  const int num_m = (p.Mk + C::TILE_M - 1) / C::TILE_M;
  const int num_n = (p.Nk + BN - 1) / BN;
  const int num_tiles = num_m * num_n;
  const int num_kb = (p.K + KB - 1) / KB;
  const int dp_tiles = num_tiles - p.sk_tiles;
  const int num_units = p.sk_tiles > 0 ? dp_tiles : p.tail_start + (num_tiles - p.tail_start) * p.split;
  constexpr int CL = PAIR ? 2 : 1;  // CTAs per cluster
  const int first_tile = static_cast<int>(blockIdx.x) / CL;
  const int tile_step = static_cast<int>(gridDim.x) / CL;
  const long long sk_iters = static_cast<long long>(p.sk_tiles) * num_kb;
  auto make_sched = [&]() {
    Sched sc;
    sc.u = first_tile;
    sc.step = tile_step;
    sc.num_units = num_units;
    sc.tail_start = p.tail_start;
    sc.split = p.split;
    sc.num_kb = num_kb;
    sc.dp_tiles = dp_tiles;
    sc.worker = first_tile;
    sc.it = p.sk_tiles > 0 ? sk_begin(first_tile, sk_iters, tile_step) : 0;
    sc.it_end = p.sk_tiles > 0 ? sk_begin(first_tile + 1, sk_iters, tile_step) : 0;
    return sc;
  };
  auto coords = [&](int tile, int& mt, int& nt) { tile_coords(tile, num_m, num_n, p.group_m, mt, nt); };
  bool aborted_here = false;

  // ------------------------------------------------ TMA producer
  // role_a: the CTA's producer (warp 0): the stage's expected bytes, A (and
  // B unless a second producer takes it), the fill count and the drain.
  // !role_a: the second producer (warp 2 + EPIW, p.two_producers): B only,
  // on the same barriers -- a thread issues a TMA box only every few
  // hundred cycles, so with an M/N-major operand (three or four boxes a
  // stage) a second thread keeps the stages coming.
  auto run_producer = [&](bool role_a) {
    {
      const bool do_a = role_a;
      const bool do_b = !role_a || AM || !p.two_producers;  // (AM: no second producer warp)
      int stage = 0;
      uint32_t phase = 0;
      long long fills = 0;
      bool ok = true;
      Sched sched = make_sched();
      int tile, kb0, kb1, v, u;
      while (ok && sched.next(tile, kb0, kb1, v, u)) {
        int mt, nt;
        coords(tile, mt, nt);
        const int row0 = mt * C::TILE_M + static_cast<int>(pr) * BM;     // this CTA's A rows
        const int col0 = nt * BN + static_cast<int>(pr) * C::B_ROWS;     // this CTA's B columns
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.budget)) {
            if (!*abort_flag) atomicOr(p.err, ERR_PRODUCER_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          uint32_t fb = full_bar(stage);
          if constexpr (AM) {
            // each CTA counts its own operands and mask slice: its transform
            // warps wait for exactly these bytes
            mbar_arrive_expect_tx(fb, C::STAGE_BYTES + C::MASK_SLOT);
          } else {
            if (role_a && (!PAIR || leader)) mbar_arrive_expect_tx(fb, (PAIR ? 2 : 1) * C::STAGE_BYTES);
            if constexpr (PAIR) fb = mapa_shared(fb, lead);  // completion counted by the pair's leader
          }
          const uint32_t sa = sbase + stage * C::STAGE_BYTES;
          const uint32_t sb = sa + C::A_BYTES;
          const int k0 = kb * KB;
          // TMA: the innermost coordinate of every box is a multiple of 64
          // elements (128 bytes): k0 for a K-major operand, row0 / col0 for
          // an M/N-major one (a K-major operand's rows are the box's outer
          // coordinate, any value: 224-wide pair tiles start B' at 112 r);
          // the stage lies below the epilogue buffers
          if (!GE_DCHECK(k0 >= 0 && k0 % 64 == 0 && row0 >= 0 && (!p.a_mn || row0 % 64 == 0) && col0 >= 0 &&
                             (!p.b_mn || col0 % 64 == 0) && (stage + 1) * C::STAGE_BYTES <= C::OFF_EPI &&
                             kb < num_kb,
                         p.err)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          auto load = [&](uint32_t dst, const CUtensorMap* map, int x, int y) {
            if constexpr (PAIR && !AM)
              tma_load_2d_pair(dst, map, fb, x, y);
            else
              tma_load_2d(dst, map, fb, x, y);
          };
          // AM: the mask words of k-rows k0.. for this CTA's A' rows row0..
          // (row0 is a multiple of 128, so the word coordinate is 16-byte aligned)
          if constexpr (AM) load(sbase + C::OFF_MASK + stage * C::MASK_SLOT, &tmZ, row0 / 32, k0);
          // K-major with two panels: one 3-D box (64 k x rows x 2 panels)
          // of a panel-indexed view of the operand.
          auto load3 = [&](uint32_t dst, const CUtensorMap* map, int y, int z) {
            if constexpr (PAIR && !AM)
              tma_load_3d_pair(dst, map, fb, 0, y, z);
            else
              tma_load_3d(dst, map, fb, 0, y, z);
          };
          // M/N-major: 64-wide chunks of KB k-rows (KB x 128 bytes each)
          constexpr uint32_t MN_CHUNK = KB * 128;
          if (!do_a) {
          } else if (!p.a_mn) {
            if constexpr (C::PANELS >= 2)
              load3(sa, &tmA, row0, C::PANELS * kb);
            else
              load(sa, &tmA, k0, row0);
          } else {
            load(sa, &tmA, row0, k0);
            load(sa + MN_CHUNK, &tmA, row0 + 64, k0);
          }
          if (!do_b) {
          } else if (!p.b_mn) {
            if constexpr (C::PANELS >= 2)
              load3(sb, &tmB, col0, C::PANELS * kb);
            else
              load(sb, &tmB, k0, col0);
          } else {
            // (an N-major B is staged in 64-wide chunks: B_ROWS a multiple of 64)
            if constexpr (C::B_ROWS % 64 == 0) {
#pragma unroll
              for (int j = 0; j < C::B_ROWS / 64; ++j) load(sb + MN_CHUNK * j, &tmB, col0 + 64 * j, k0);
            }
          }
          ++fills;
#ifdef GE_DEBUG
          if (role_a && stage < 8) dbg_fills[stage] = dbg_fills[stage] + 1u;
#endif
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: every issued load must land before the CTA may exit (the
      // second producer's loads land on the same barriers).
      if (!role_a) {
        if (!ok) {
          const long long t0 = clock64();
          while (clock64() - t0 < 100000LL) {
          }
        }
      } else if (!PAIR || leader || AM) {
        for (int s = 0; s < C::STAGES; ++s) {
          if (fills > s) {
            const long long last = s + (long long)C::STAGES * ((fills - 1 - s) / C::STAGES);
            const uint32_t par = static_cast<uint32_t>((last / C::STAGES) & 1);
            if (!mbar_wait_bounded(full_bar(s), par, never, p.budget)) atomicOr(p.err, ERR_DRAIN_TIMEOUT);
          }
        }
      } else if (!ok) {
        // The odd CTA's loads are counted on the leader's barriers; after an
        // abort give any copy still in flight time to land (~50 us).
        const long long t0 = clock64();
        while (clock64() - t0 < 100000LL) {
        }
      }
      if (role_a) aborted_here = !ok;
    }
  };
  if (warp == 0) {
    if (lane == 0) run_producer(true);
  } else if (!AM && warp == 2 + EPIW) {
    if (lane == 0 && p.two_producers) run_producer(false);
  } else if (warp == 1) {
    if (lane == 0 && (!PAIR || leader)) {
      // ------------------------------------------------ MMA issuer
      const uint32_t idesc = idesc_f16_f32(C::TILE_M, BN, p.a_mn, p.b_mn, p.bf16 ? 1u : 0u);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
#ifdef GE_DEBUG
      unsigned int uses[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // stages consumed so far
#endif
      Sched sched = make_sched();
      int tile, kb0, kb1, v, u;
      while (ok && sched.next(tile, kb0, kb1, v, u)) {
        if (!GE_DCHECK(acc * BN + BN <= C::TMEM_COLS && kb0 < kb1, p.err)) {
          *abort_flag = 1;
          break;
        }
        if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.budget)) {
          if (!*abort_flag) atomicOr(p.err, ERR_MMA_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = kb0; kb < kb1; ++kb) {
#ifdef GE_DEBUG
          // the fills of this stage the producer issued so far, less the
          // uses: 0 (not yet refilled) or 1; 2 would be a phase the parity
          // wait cannot tell from the one it waits for
          if (stage < 8) {  // (pairs: the leader's own producer's fills)
            const unsigned int ahead = dbg_fills[stage] - uses[stage];
            if (!GE_DCHECK(ahead <= 1u, p.err)) {
              *abort_flag = 1;
              ok = false;
              break;
            }
          }
          if (stage < 8) ++uses[stage];
#endif
          bool landed;
          if constexpr (AM)  // masked by both CTAs' transform warps
            landed = PAIR ? mbar_wait_bounded_cluster(xform_bar(stage), phase, abort_flag, p.budget)
                          : mbar_wait_bounded(xform_bar(stage), phase, abort_flag, p.budget);
          else
            landed = mbar_wait_bounded(full_bar(stage), phase, abort_flag, p.budget);
          if (!landed) {
            if (!*abort_flag) atomicOr(p.err, ERR_MMA_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = sbase + stage * C::STAGE_BYTES;
          const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
          for (int k = 0; k < KB / 16; ++k) {
            // K-major: the 16-wide k step is 32 bytes inside the 128-byte
            // swizzle row of its panel (panels of rows x 128 bytes follow
            // one another); MN-major: 16 k-rows of 128 bytes = 2 KB, the
            // 64-wide chunks KB x 128 bytes apart.
            const uint32_t pk = static_cast<uint32_t>(k >> 2), wk = static_cast<uint32_t>(k & 3);
            const uint64_t ad = p.a_mn ? smem_desc_sw128(sa + 2048u * k, KB * 128u, 1024u)
                                       : smem_desc_sw128(sa + pk * (BM * 128u) + 32u * wk, 16u, 1024u);
            const uint64_t bd = p.b_mn ? smem_desc_sw128(sb + 2048u * k, KB * 128u, 1024u)
                                       : smem_desc_sw128(sb + pk * (C::B_ROWS * 128u) + 32u * wk, 16u, 1024u);
            if constexpr (PAIR)
              tc_mma_f16_pair(d_tmem, ad, bd, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
            else
              tc_mma_f16(d_tmem, ad, bd, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
          }
          // frees the stage (in both CTAs of a pair) once these MMAs retire
          if constexpr (PAIR)
            tc_commit_pair_mc(empty_bar(stage), 0x3);
          else
            tc_commit(empty_bar(stage));
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        // accumulator ready for the epilogue (of both CTAs of a pair)
        if constexpr (PAIR)
          tc_commit_pair_mc(tfull_bar(acc), static_cast<uint16_t>(0x3u << lead));
        else
          tc_commit(tfull_bar(acc));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Drain: all MMAs issued by this thread retire before TMEM is freed.
      if constexpr (PAIR)
        tc_commit_pair_mc(drain_bar, static_cast<uint16_t>(0x1u << lead));
      else
        tc_commit(drain_bar);
      if (!mbar_wait_bounded(drain_bar, 0u, never, p.budget)) atomicOr(p.err, ERR_DRAIN_TIMEOUT);
    }
  } else if (AM && warp >= 2 + EPIW) {
    // ------------------------------------------ A-operand mask (AM only)
    // A' is M-major: a stage holds this CTA's BM = 128 rows as two 8 KB
    // chunks of BK = 64 k-rows x 64 m (128 bytes, 128-byte swizzle: the
    // 16-byte unit u of k-row r sits at unit u ^ (r & 7)). Thread t owns the
    // 8 m of unit (t >> 3) on the k-rows r = (t & 7) + 8i, so its physical
    // unit is the same on every row, and it keeps their masked fp32 sums.
    const int xt = static_cast<int>(threadIdx.x) - 32 * (2 + EPIW);
    const int xunit = xt >> 3, ph = xt & 7;
    const int chunk = xunit >> 3, uu = xunit & 7;
    const uint32_t a_off = 8192u * chunk + 16u * static_cast<uint32_t>(uu ^ ph);
    const int wsel = 2 * chunk + (uu >> 2);  // mask word of these 8 m (of the row's 4)
    const int bsh = 8 * (uu & 3);
    const bool bf16 = p.bf16 != 0;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    Sched sched = make_sched();
    int tile, kb0, kb1, v, u;
    while (ok && sched.next(tile, kb0, kb1, v, u)) {
      int mt, nt;
      coords(tile, mt, nt);
      const bool want_bg = p.bg_partials != nullptr && nt == 0;
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
      for (int kb = kb0; kb < kb1; ++kb) {
        int okw = 1;
        if (lane == 0) okw = mbar_wait_bounded(full_bar(stage), phase, abort_flag, p.budget) ? 1 : 0;
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) {
          if (lane == 0) {
            if (!*abort_flag) atomicOr(p.err, ERR_XFORM_TIMEOUT);
            *abort_flag = 1;
          }
          ok = false;
          break;
        }
        uint8_t* abase = smem + stage * C::STAGE_BYTES + a_off;
        const uint32_t* mrow = reinterpret_cast<const uint32_t*>(smem + C::OFF_MASK + stage * C::MASK_SLOT) + wsel;
#pragma unroll
        for (int i = 0; i < BK / 8; ++i) {
          const int r = ph + 8 * i;
          const uint32_t bits = (mrow[4 * r] >> bsh) & 0xFFu;
          uint4* cell = reinterpret_cast<uint4*>(abase + 128 * r);
          const uint4 val = *cell;
          uint32_t w[4] = {val.x, val.y, val.z, val.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint32_t keep = ((bits >> (2 * t)) & 1u ? 0x0000FFFFu : 0u) |
                                  ((bits >> (2 * t + 1)) & 1u ? 0xFFFF0000u : 0u);
            w[t] &= keep;  // a cleared element is +0 in either type
            if (want_bg) {
              const float2 f = to_f32x2(bf16, w[t]);
              acc[2 * t] += f.x;
              acc[2 * t + 1] += f.y;
            }
          }
          *cell = make_uint4(w[0], w[1], w[2], w[3]);
        }
        // the masked tile must be visible to the tensor core (async proxy)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (PAIR && !leader)
            mbar_arrive_remote(mapa_shared(xform_bar(stage), lead));
          else
            mbar_arrive(xform_bar(stage));
        }
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (want_bg) {
        // the 8 k-row phases of each unit are 8 adjacent lanes: a fixed tree
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 1);
          acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 2);
          acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 4);
        }
        if (ph == 0) {
          const int m0 = mt * C::TILE_M + static_cast<int>(pr) * BM + 64 * chunk + 8 * uu;
          const int piece = v >= 0 ? v % p.split : 0;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (m0 + e < p.Mk) {
              p.bg_partials[static_cast<long long>(piece) * p.Mk + m0 + e] = acc[e];
              if (v < 0)  // a whole tile: the other pieces' rows hold nothing
                for (int sp = 1; sp < p.split; ++sp) p.bg_partials[static_cast<long long>(sp) * p.Mk + m0 + e] = 0.0f;
            }
          }
        }
      }
    }
  } else {
    // -------------------------------------------------- epilogue warps
    const int q = warp & 3;           // TMEM lane quarter this warp may access
    const int hh = (warp - 2) >> 2;   // which of the quarter's warps: slabs hh, hh + HALVES, ...
    uint8_t* stg = smem + C::OFF_EPI + (warp - 2) * 2 * EPI_BUF_BYTES;
    constexpr bool backward = EPI == EPI_DRELU_BGRAD || EPI == EPI_DGELU_BGRAD;
    constexpr bool has_bias = EPI != EPI_NONE && !backward;
    const bool bf16 = p.bf16 != 0;
    const unsigned short* bias16 = reinterpret_cast<const unsigned short*>(p.bias);
    int acc = 0;
    uint32_t acc_phase = 0;
    int nstore = 0;
    // stream-K: the value this launch's completion flags carry (the epoch
    // word changes only after every CTA of the launch has finished)
    const unsigned int sk_mark = p.sk_tiles > 0 ? *reinterpret_cast<volatile unsigned int*>(p.sk_sync) + 1u : 0u;
    Sched sched = make_sched();
    int tile, kb0, kb1, v, u;
    bool warm_code = true;  // the first tile epilogue still has its dry pass to run
    while (sched.next(tile, kb0, kb1, v, u)) {
      int mt, nt;
      coords(tile, mt, nt);
      const int rbase = mt * C::TILE_M + static_cast<int>(pr) * BM + q * 32;  // warp's first row of D'
      const int grow = rbase + lane;                                          // this thread's row
      // DGELU_BGRAD's z / BIAS_RESIDUAL's residual: the first slab is
      // requested before the wait for the accumulator, each later one while
      // the slab before it is processed.
      const bool needs_z = v < 0 && (EPI == EPI_DGELU_BGRAD || EPI == EPI_BIAS_RESIDUAL);
      // Ask L2 for this thread's row segment of the next unit's per-element
      // input (z / residual / mask) now, a whole tile ahead of its use: the
      // slab loads then hit L2 instead of waiting on DRAM.
      // (A bulk prefetch needs a 16-byte aligned start: the row pitches are
      // multiples of 16 bytes, so only the base pointer is checked.)
      const void* pf_base = EPI == EPI_DRELU_BGRAD ? static_cast<const void*>(p.aux) : p.zaux;
      if ((EPI == EPI_DGELU_BGRAD || EPI == EPI_BIAS_RESIDUAL || EPI == EPI_DRELU_BGRAD) &&
          (reinterpret_cast<uintptr_t>(pf_base) & 15u) == 0) {
        for (int k = (u == first_tile ? 0 : 1); k < 2 && hh == 0 && u >= 0; ++k) {
          const int un = u + k * tile_step;
          if (un >= num_units) break;
          int tn, kb0n, kb1n, vn, mtn, ntn;
          unit_info(un, p.tail_start, p.split, num_kb, tn, kb0n, kb1n, vn);
          if (vn >= 0) continue;
          coords(tn, mtn, ntn);
          const int rown = mtn * C::TILE_M + static_cast<int>(pr) * BM + q * 32 + lane;
          const int c0 = ntn * BN;
          const int ncols = min(BN, p.Nk - c0);
          if (rown < p.Mk && ncols > 0) {
            if (EPI == EPI_DRELU_BGRAD)
              bulk_prefetch_l2(p.aux + static_cast<long long>(rown) * p.ld_aux + (c0 >> 5),
                               static_cast<uint32_t>((((ncols + 31) >> 5) * 4 + 15) & ~15));
            else
              bulk_prefetch_l2(p.zaux + static_cast<long long>(rown) * p.ld_zaux + c0,
                               static_cast<uint32_t>((ncols * 2 + 15) & ~15));
          }
        }
      }
      uint32_t zw[16];
      if (needs_z) load_slab16(p, grow, nt * BN + 32 * hh, zw);
      // The bias is requested before the wait as well, the first slab's now
      // and each later one's a slab ahead, and kept as loaded (converted at
      // use, so a load in flight stalls nothing): per row, this thread's
      // value; per column, with a 16-byte aligned bias, the slab's 32 raw
      // values in every lane (four 16-byte loads of one address, a
      // broadcast); otherwise, and for a slab that runs past Nk, lane l
      // holds column 32c + l and the 32 values are broadcast by shuffles.
      float brow = 0.0f;
      if (has_bias && !p.bias_per_col && grow < p.Mk) brow = to_f32(bf16, bias16[grow]);
      const bool bias_cols = has_bias && p.bias_per_col;
      const bool bias_vec = bias_cols && (reinterpret_cast<uintptr_t>(bias16) & 15u) == 0;
      auto bias_lane = [&](int gc) -> unsigned short {
        return bias_cols && !bias_vec && gc < p.Nk ? bias16[gc] : static_cast<unsigned short>(0);
      };
      auto bias_run = [&](int gc, uint4 (&b)[4]) {
        if (bias_vec && gc + 32 <= p.Nk) {
#pragma unroll
          for (int i = 0; i < 4; ++i) b[i] = __ldg(reinterpret_cast<const uint4*>(bias16 + gc) + i);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) b[i] = make_uint4(0u, 0u, 0u, 0u);
        }
      };
      // (with eight epilogue warps a thread has 168 registers: the slab's
      // run is then loaded at the slab's start, behind its TMEM load)
      constexpr bool kBiasAhead = EPIW == 4;
      uint4 bq[4];
      if constexpr (kBiasAhead) bias_run(nt * BN + 32 * hh, bq);
      unsigned short bl = bias_lane(nt * BN + 32 * hh + lane);
      // Stream-K finisher: the workers sk_w0 .. sk_w1 - 1 hold the rest of
      // this tile's k-range (their first segments, spilled early in their
      // ranges); wait until this warp's rows of each of their slots are
      // complete (the flag written by the same warp of the same CTA rank).
      const bool finish = v == kFinish;
      int sk_w0 = 0, sk_w1 = 0;
      if (finish) {
        const long long tile_end = static_cast<long long>(tile - dp_tiles + 1) * num_kb;
        sk_w0 = first_tile + 1;
        sk_w1 = sk_w0;
        while (sk_w1 < tile_step && sk_begin(sk_w1, sk_iters, tile_step) < tile_end) ++sk_w1;
        int fok = 1;
        if (lane == 0) {
          for (int wq = sk_w0; wq < sk_w1 && fok; ++wq) {
            if (sk_begin(wq + 1, sk_iters, tile_step) == sk_begin(wq, sk_iters, tile_step)) continue;  // no piece
            const unsigned int* flag =
                p.sk_sync + 2 + (static_cast<long long>(wq) * CL + static_cast<int>(pr)) * EPIW + (warp - 2);
            if (ld_acquire_gpu(flag) == sk_mark) continue;
            const long long t0 = clock64();
            while (ld_acquire_gpu(flag) != sk_mark) {
              if (*abort_flag || clock64() - t0 > p.budget) {
                fok = 0;
                break;
              }
            }
          }
          if (!fok) {
            if (!*abort_flag) atomicOr(p.err, ERR_PEER_TIMEOUT);
            *abort_flag = 1;
          }
        }
        fok = __shfl_sync(0xffffffffu, fok, 0);
        if (!fok) break;
        // every lane acquires the flags too (its loads of the pieces come
        // after), then asks the first slab's pieces into L1
        for (int wq = sk_w0; wq < sk_w1; ++wq)
          if (sk_begin(wq + 1, sk_iters, tile_step) != sk_begin(wq, sk_iters, tile_step))
            (void)ld_acquire_gpu(p.sk_sync + 2 + (static_cast<long long>(wq) * CL + static_cast<int>(pr)) * EPIW + (warp - 2));
      }
      // The pieces of slab c of this warp: 4 KB per worker slot (8 chunks of
      // 512 bytes); lane l asks line l of each into L1 a slab ahead of use.
      auto piece_chunks = [&](int wq, int c) -> const uint4* {
        return reinterpret_cast<const uint4*>(
                   p.partials + (static_cast<long long>(wq) * C::TILE_M + static_cast<int>(pr) * BM) * BN) +
               static_cast<long long>((q * (BN / 32) + c) * 8) * 32;
      };
      auto piece_prefetch = [&](int c) {
        for (int wq = sk_w0; wq < sk_w1; ++wq)
          if (sk_begin(wq + 1, sk_iters, tile_step) != sk_begin(wq, sk_iters, tile_step))
            prefetch_l1(piece_chunks(wq, c) + 8 * lane);
      };
      if (finish) piece_prefetch(hh);
      // The worker's first tile epilogue (v < 0) is preceded by a dry pass
      // over its first slab while the accumulator is still being computed:
      // the same instructions (the pass loop is not unrolled) without TMEM
      // loads or memory side effects, so that the real pass finds them in
      // the instruction cache (measured: the first slab of a CTA took ~11k
      // cycles, a later one ~2.3k; the activation alone 5.4k vs 0.85k).
      bool failed = false;
#pragma unroll 1
      for (int pass = (warm_code && v < 0) ? 0 : 1; pass < 2; ++pass) {
        const bool dry = pass == 0;
        if (!dry) {
          int ok = 1;
          if (lane == 0) ok = mbar_wait_bounded(tfull_bar(acc), acc_phase, abort_flag, p.budget) ? 1 : 0;
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) {
            if (lane == 0) {
              if (!*abort_flag) atomicOr(p.err, ERR_EPILOGUE_TIMEOUT);
              *abort_flag = 1;
            }
            failed = true;
            break;
          }
          tc_fence_after();
          if (v >= 0) {
            // Split-K unit: spill the fp32 accumulator rows to its piece of
            // the workspace ([TILE_M][BN], read row-wise by the fixup kernel,
            // which adds the pieces and applies the epilogue). Each 32 x 32
            // slab goes through the warp's staging buffer (4 KB: 16-byte
            // chunk j of row r at chunk j ^ (r & 7)) so that every global
            // store covers 4 rows x 128 bytes; written straight from the
            // lanes (a row each, 16 bytes 1 KB apart) the spill of a 256 x
            // 256 tile took ~9 us. A stream-K segment (u < 0) goes to the
            // worker's slot, which holds each warp's slabs lane-interleaved
            // (chunk i of lane l of slab c at ((q * BN / 32 + c) * 8 + i) *
            // 32 + l in the CTA's half): every store and the finisher's every
            // load covers 512 contiguous bytes.
            (void)GE_DCHECK(u >= 0 || v == first_tile, p.err);
            float* prow0 = p.partials + (static_cast<long long>(v) * C::TILE_M + static_cast<int>(pr) * BM + q * 32) * BN;
            uint4* slot = reinterpret_cast<uint4*>(p.partials + (static_cast<long long>(v) * C::TILE_M +
                                                                 static_cast<int>(pr) * BM) * BN);
            if (u >= 0) {  // the staging buffer is free once this warp's stores have read it
              if (lane == 0) bulk_wait_group_read<0>();
              __syncwarp();
            }
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
#pragma unroll 1
            for (int c = hh; c < BN / 32; c += C::HALVES) {
              uint32_t vv[32];
              tmem_ld_32x32b_x32(t_row + 32u * c, vv);
              tmem_ld_wait();
              if (u < 0) {
                uint4* dst = slot + static_cast<long long>((q * (BN / 32) + c) * 8) * 32 + lane;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  dst[32 * i] = make_uint4(vv[4 * i], vv[4 * i + 1], vv[4 * i + 2], vv[4 * i + 3]);
              } else {
                uint4* st4 = reinterpret_cast<uint4*>(stg);
                __syncwarp();  // the previous slab has been read back
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  st4[lane * 8 + (j ^ (lane & 7))] = make_uint4(vv[4 * j], vv[4 * j + 1], vv[4 * j + 2], vv[4 * j + 3]);
                __syncwarp();
                // lane l: chunk l & 7 of rows 4i + l / 8
                const int ch = lane & 7;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const int r = 4 * i + (lane >> 3);
                  reinterpret_cast<uint4*>(prow0 + static_cast<long long>(r) * BN + c * 32)[ch] = st4[r * 8 + (ch ^ (r & 7))];
                }
              }
            }
            if (u < 0) {
              // this warp's rows of the slot are complete: publish them
              __threadfence();
              __syncwarp();
              if (lane == 0)
                st_release_gpu(p.sk_sync + 2 + static_cast<long long>(blockIdx.x) * EPIW + (warp - 2), sk_mark);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (PAIR && !leader)
                mbar_arrive_remote(mapa_shared(tempty_bar(acc), lead));
              else
                mbar_arrive(tempty_bar(acc));
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
            break;
          }
        }  // !dry
        float bg_row = 0.0f;  // D*_BGRAD, bias per D' row: this tile's row sum
        float st_n = 0.0f, st_mean = 0.0f, st_m2 = 0.0f;  // BIAS_RESIDUAL statistics of this row
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                               static_cast<uint32_t>(acc * BN);
        // the last n-tile also writes the mask's zero padding words up to
        // the next multiple of 128 columns (a tile narrower than 128 -- 224
        // wide -- can end before it)
        const int c_end = (EPI == EPI_RELU_AUX_BIAS && nt == num_n - 1)
                              ? max(BN / 32, ((((p.Nk + 127) & ~127) - nt * BN) + 31) / 32)
                              : BN / 32;
#pragma unroll 1
        for (int c = hh; c < c_end; c += C::HALVES) {
          if (dry && c != hh) break;
          const int gcol0 = nt * BN + c * 32;
          if (gcol0 >= p.Nk) {
            // Past the end of the row: only the mask's zero padding words
            // (rows padded to 128 columns) remain to be written.
            if (!dry && EPI == EPI_RELU_AUX_BIAS && grow < p.Mk && gcol0 < ((p.Nk + 127) & ~127))
              p.aux[static_cast<long long>(grow) * p.ld_aux + (gcol0 >> 5)] = 0u;
            continue;
          }
          // DRELU_BGRAD: the slab's mask word is requested before the TMEM load
          // so the two latencies overlap.
          uint32_t mword = 0;
          if (!dry && EPI == EPI_DRELU_BGRAD && grow < p.Mk)
            mword = p.aux[static_cast<long long>(grow) * p.ld_aux + (gcol0 >> 5)];
          uint32_t znext[16];
          if (!dry && needs_z && c + C::HALVES < BN / 32) load_slab16(p, grow, gcol0 + 32 * C::HALVES, znext);
          uint4 bq_next[4];
          if constexpr (kBiasAhead)
            bias_run(gcol0 + 32 * C::HALVES, bq_next);
          else
            bias_run(gcol0, bq);
          if (finish && !dry && c + C::HALVES < BN / 32) piece_prefetch(c + C::HALVES);
          const unsigned short bl_next = bias_lane(gcol0 + 32 * C::HALVES + lane);
          uint32_t v[32];
          (void)GE_DCHECK(acc * BN + 32 * c + 32 <= C::TMEM_COLS && gcol0 % 32 == 0 && rbase % 32 == 0 &&
                        (p.aux == nullptr || (gcol0 >> 5) < p.ld_aux),
                    p.err);
          if (dry) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0u;
          } else {
            tmem_ld_32x32b_x32(t_row + 32u * c, v);
            tmem_ld_wait();
          }
          if (finish && !dry) {
            // add the rest of the tile's k-range, slot by slot in k order
#pragma unroll 1
            for (int wq = sk_w0; wq < sk_w1; ++wq) {
              if (sk_begin(wq + 1, sk_iters, tile_step) == sk_begin(wq, sk_iters, tile_step)) continue;
              const uint4* src = piece_chunks(wq, c) + lane;
              uint4 pv[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) pv[i] = src[32 * i];  // (in L1: asked for a slab ahead)
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                v[4 * i] = __float_as_uint(__uint_as_float(v[4 * i]) + __uint_as_float(pv[i].x));
                v[4 * i + 1] = __float_as_uint(__uint_as_float(v[4 * i + 1]) + __uint_as_float(pv[i].y));
                v[4 * i + 2] = __float_as_uint(__uint_as_float(v[4 * i + 2]) + __uint_as_float(pv[i].z));
                v[4 * i + 3] = __float_as_uint(__uint_as_float(v[4 * i + 3]) + __uint_as_float(pv[i].w));
              }
            }
          }
          float bcol[32];
          if (bias_vec && gcol0 + 32 <= p.Nk) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 b = bq[i];
              const float2 f0 = to_f32x2(bf16, b.x), f1 = to_f32x2(bf16, b.y);
              const float2 f2 = to_f32x2(bf16, b.z), f3 = to_f32x2(bf16, b.w);
              bcol[8 * i] = f0.x;
              bcol[8 * i + 1] = f0.y;
              bcol[8 * i + 2] = f1.x;
              bcol[8 * i + 3] = f1.y;
              bcol[8 * i + 4] = f2.x;
              bcol[8 * i + 5] = f2.y;
              bcol[8 * i + 6] = f3.x;
              bcol[8 * i + 7] = f3.y;
            }
          } else if (bias_cols) {
            const unsigned short b1 =
                bias_vec ? (gcol0 + lane < p.Nk ? bias16[gcol0 + lane] : static_cast<unsigned short>(0)) : bl;
            const float blf = to_f32(bf16, b1);
#pragma unroll
            for (int j = 0; j < 32; ++j) bcol[j] = __shfl_sync(0xffffffffu, blf, j);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) bcol[j] = brow;  // the row's bias (0 without one)
          }
          if (!dry) {
            bl = bl_next;
            if constexpr (kBiasAhead) {
#pragma unroll
              for (int i = 0; i < 4; ++i) bq[i] = bq_next[i];
            }
          }
          uint32_t packed[16];
          uint32_t zpacked[16];
          uint32_t bits = 0;
          if (backward) {
            // DRELU_BGRAD: dZ = dH where the forward mask bit is set, else +0.
            // DGELU_BGRAD: dZ = dH * gelu'(z) with z the stored pre-activation.
            // The fp32 values (before rounding) feed the bias-gradient sums;
            // columns past Nk contribute 0.
            float zm[32];
            if (EPI == EPI_DRELU_BGRAD) {
              uint32_t w = mword;
              if (p.Nk - gcol0 < 32) w &= (1u << (p.Nk - gcol0)) - 1u;
#pragma unroll
              for (int j = 0; j < 32; ++j) zm[j] = ((w >> j) & 1u) ? __uint_as_float(v[j]) : 0.0f;
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float2 z = to_f32x2(bf16, zw[j]);
                zm[2 * j] = gcol0 + 2 * j < p.Nk ? __uint_as_float(v[2 * j]) * gelu_tanh_grad(z.x) : 0.0f;
                zm[2 * j + 1] =
                    gcol0 + 2 * j + 1 < p.Nk ? __uint_as_float(v[2 * j + 1]) * gelu_tanh_grad(z.y) : 0.0f;
              }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) packed[j] = pack2(bf16, zm[2 * j], zm[2 * j + 1]);
            if (p.bias_per_col) {
              // bgrad indexes D' columns: reduce the 32 rows of this warp for
              // each of its 32 columns (lane l ends with column gcol0 + l).
#pragma unroll
              for (int off = 16; off >= 1; off >>= 1) {
                const bool upper = (lane & off) != 0;
#pragma unroll
                for (int i = 0; i < off; ++i) {
                  const float send = upper ? zm[i] : zm[i + off];
                  const float keep = upper ? zm[i + off] : zm[i];
                  zm[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
              }
              if (!dry && rbase < p.Mk && gcol0 + lane < p.Nk)
                p.bg_partials[static_cast<long long>(rbase >> 5) * p.Nk + gcol0 + lane] = zm[0];
            } else {
              float srow = 0.0f;
#pragma unroll
              for (int j = 0; j < 32; ++j) srow += zm[j];
              bg_row += srow;
            }
          } else if (EPI == EPI_BIAS_RESIDUAL) {
            // h = acc + bias + residual, stored once; with nstats the slab's
            // exact mean and squared deviations (two passes over registers)
            // are merged into the tile's running pair by Chan's formula.
            float hv[32];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float2 r = to_f32x2(bf16, zw[j]);
              hv[2 * j] = __uint_as_float(v[2 * j]) + bcol[2 * j] + r.x;
              hv[2 * j + 1] = __uint_as_float(v[2 * j + 1]) + bcol[2 * j + 1] + r.y;
              packed[j] = pack2(bf16, hv[2 * j], hv[2 * j + 1]);
            }
            if (p.nstats) {
              const int nvalid = p.Nk - gcol0 < 32 ? p.Nk - gcol0 : 32;
              float s = 0.0f;
#pragma unroll
              for (int j = 0; j < 32; ++j) s += j < nvalid ? hv[j] : 0.0f;
              const float nb = static_cast<float>(nvalid);
              const float m = s / nb;
              float q = 0.0f;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float d = j < nvalid ? hv[j] - m : 0.0f;
                q = fmaf(d, d, q);
              }
              const float nn = st_n + nb;
              const float delta = m - st_mean;
              st_mean = fmaf(delta, nb / nn, st_mean);
              st_m2 += fmaf(delta * delta, st_n * nb / nn, q);
              st_n = nn;
            }
          } else {
            bits = epilogue_slab<EPI>(v, bcol, packed, zpacked, bf16);
          }
          (void)GE_DCHECK(!dry || nstore == 0, p.err);  // no store of this CTA in flight
          store_slab(packed, &tmD, reinterpret_cast<unsigned short*>(p.D), p.ldd, gcol0, rbase, grow,
                     p.Mk, p.Nk, stg, nstore, lane, p.err, dry);
          if (EPI == EPI_GELU_AUX_BIAS)
            store_slab(zpacked, &tmZ, p.zaux, p.ld_zaux, gcol0, rbase, grow, p.Mk, p.Nk, stg, nstore, lane, p.err,
                       dry);
          if (!dry && EPI == EPI_RELU_AUX_BIAS && grow < p.Mk) {
            if (p.Nk - gcol0 < 32) bits &= (1u << (p.Nk - gcol0)) - 1u;
            p.aux[static_cast<long long>(grow) * p.ld_aux + (gcol0 >> 5)] = bits;
          }
          if (needs_z && !dry) {
#pragma unroll
            for (int j = 0; j < 16; ++j) zw[j] = znext[j];
          }
        }
        if (dry) continue;
        if (backward && !p.bias_per_col && grow < p.Mk)
          p.bg_partials[static_cast<long long>(C::HALVES * nt + hh) * p.Mk + grow] = bg_row;
        if (EPI == EPI_BIAS_RESIDUAL && p.nstats && grow < p.Mk)
          p.nstats[static_cast<long long>(C::HALVES * nt + hh) * p.Mk + grow] = make_float2(st_mean, st_m2);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          // this warp's share of the accumulator is free (the pair's MMA
          // issuer counts the arrivals of both CTAs' epilogue warps)
          if (PAIR && !leader)
            mbar_arrive_remote(mapa_shared(tempty_bar(acc), lead));
          else
            mbar_arrive(tempty_bar(acc));
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }  // pass
      if (v < 0) warm_code = false;
      if (failed) break;
    }
    // The stores must have read their staging buffers before the CTA's
    // shared memory goes away; their global writes complete with the grid.
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
  }
  (void)aborted_here;

  __syncwarp();
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync();  // neither CTA leaves while its peer may still touch it
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, C::TMEM_ALLOC);
    else
      tmem_dealloc(tmem_base, C::TMEM_ALLOC);
  }
  if (p.sk_tiles > 0 && threadIdx.x == 0) {
    // The last CTA of the launch to get here moves the epoch on, so the
    // next launch's flags carry a value that none written so far has.
    __threadfence();
    const unsigned int done = atomicAdd(p.sk_sync + 1, 1u);
    if (done == gridDim.x - 1) {
      atomicExch(p.sk_sync + 1, 0u);
      __threadfence();
      atomicAdd(p.sk_sync, 1u);
    }
  }
}

template <int EPI, int BN, bool PAIR, int EPIW, bool AM = false, int KB = 64>
cudaError_t launch_impl(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmD,
                        const CUtensorMap& tmZ, const GemmArgs& args, int grid, cudaStream_t stream) {
  using C = Cfg<BN, PAIR, EPIW, AM, KB>;
  static std::atomic<bool> configured[64] = {};  // the attribute is set once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(tc_gemm_kernel<EPI, BN, PAIR, EPIW, AM, KB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if constexpr (PAIR) {
      e = cudaFuncSetAttribute(tc_gemm_kernel<EPI, BN, PAIR, EPIW, AM, KB>, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
      cudaGetLastError();
    }
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(C::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if constexpr (PAIR) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  e = cudaLaunchKernelEx(&cfg, tc_gemm_kernel<EPI, BN, PAIR, EPIW, AM, KB>, tmA, tmB, tmD, tmZ, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int EPI, int EPIW>
cudaError_t launch_width(int block_n, int pair, const CUtensorMap& tmA, const CUtensorMap& tmB,
                         const CUtensorMap& tmD, const CUtensorMap& tmZ, const GemmArgs& args, int grid,
                         cudaStream_t stream) {
  if constexpr (EPIW == 4 && EPI == EPI_NONE) {
    if (args.amask) {  // four epilogue warps, no epilogue arithmetic
      if (pair) {
        if (block_n == 256) return launch_impl<EPI, 256, true, 4, true>(tmA, tmB, tmD, tmZ, args, grid, stream);
        return launch_impl<EPI, 128, true, 4, true>(tmA, tmB, tmD, tmZ, args, grid, stream);
      }
      if (block_n == 256) return launch_impl<EPI, 256, false, 4, true>(tmA, tmB, tmD, tmZ, args, grid, stream);
      return launch_impl<EPI, 128, false, 4, true>(tmA, tmB, tmD, tmZ, args, grid, stream);
    }
  } else {
    if (args.amask) return cudaErrorInvalidValue;
  }
  if (block_n == 224) {  // 256 x 224 pair tiles, K-major B' only (112 rows a CTA)
    if (!pair || args.b_mn) return cudaErrorInvalidValue;
    if (args.kb == 128) return launch_impl<EPI, 224, true, EPIW, false, 128>(tmA, tmB, tmD, tmZ, args, grid, stream);
    return launch_impl<EPI, 224, true, EPIW>(tmA, tmB, tmD, tmZ, args, grid, stream);
  }
  if (args.kb == 128) {  // stages of two panels (64 KB at most a stage)
    if (pair) {
      if (block_n == 256) return launch_impl<EPI, 256, true, EPIW, false, 128>(tmA, tmB, tmD, tmZ, args, grid, stream);
      return launch_impl<EPI, 128, true, EPIW, false, 128>(tmA, tmB, tmD, tmZ, args, grid, stream);
    }
    if (block_n == 128) return launch_impl<EPI, 128, false, EPIW, false, 128>(tmA, tmB, tmD, tmZ, args, grid, stream);
    return cudaErrorInvalidValue;
  }
  if (pair) {
    if (block_n == 256) return launch_impl<EPI, 256, true, EPIW>(tmA, tmB, tmD, tmZ, args, grid, stream);
    return launch_impl<EPI, 128, true, EPIW>(tmA, tmB, tmD, tmZ, args, grid, stream);
  }
  if (block_n == 256) return launch_impl<EPI, 256, false, EPIW>(tmA, tmB, tmD, tmZ, args, grid, stream);
  return launch_impl<EPI, 128, false, EPIW>(tmA, tmB, tmD, tmZ, args, grid, stream);
}

// Largest number of CTA pairs of the pair kernel that can be resident.
template <int BN, int EPIW>
int max_pairs(int num_sms) {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return num_sms / 2;
  }
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  cudaFuncSetAttribute(tc_gemm_kernel<EPI_NONE, BN, true, EPIW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       Cfg<BN, true, EPIW>::SMEM_BYTES);
  cudaGetLastError();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms & ~1), 1, 1);
  cfg.blockDim = dim3(Cfg<BN, true, EPIW>::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg<BN, true, EPIW>::SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel<EPI_NONE, BN, true, EPIW>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = num_sms / 2;
  }
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

}  // namespace

// The kernels of one epilogue code: picks the instantiation for the tile
// width, pair mode, epilogue width and k-values per stage of `args`.
template <int EPI>
cudaError_t launch_tc_gemm_epi(int block_n, int pair, int epi_warps, const CUtensorMap& tmA, const CUtensorMap& tmB,
                               const CUtensorMap& tmD, const CUtensorMap& tmZ, const GemmArgs& args, int grid,
                               cudaStream_t stream) {
  if (epi_warps == 8) return launch_width<EPI, 8>(block_n, pair, tmA, tmB, tmD, tmZ, args, grid, stream);
  return launch_width<EPI, 4>(block_n, pair, tmA, tmB, tmD, tmZ, args, grid, stream);
}

}  // namespace ge
