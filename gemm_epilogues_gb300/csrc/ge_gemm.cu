// ge_gemm.cu -- host side of the tensor-core GEMM: the split-K fixup kernel
// and its launch, and the dispatch of a launch to the kernels of the plan's
// epilogue code (instantiated one epilogue per translation unit,
// ge_gemm_epi_*.cu; the kernel itself is in ge_gemm_kernel.cuh).
#include "ge_gemm_kernel.cuh"

namespace ge {

extern template cudaError_t launch_tc_gemm_epi<EPI_NONE>(int, int, int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                   const GemmArgs&, int, cudaStream_t);
extern template cudaError_t launch_tc_gemm_epi<EPI_BIAS>(int, int, int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                   const GemmArgs&, int, cudaStream_t);
extern template cudaError_t launch_tc_gemm_epi<EPI_RELU_BIAS>(int, int, int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                   const GemmArgs&, int, cudaStream_t);
extern template cudaError_t launch_tc_gemm_epi<EPI_GELU_BIAS>(int, int, int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                   const GemmArgs&, int, cudaStream_t);
extern template cudaError_t launch_tc_gemm_epi<EPI_GELU_ERF_BIAS>(int, int, int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                   const GemmArgs&, int, cudaStream_t);
extern template cudaError_t launch_tc_gemm_epi<EPI_RELU_AUX_BIAS>(int, int, int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                   const GemmArgs&, int, cudaStream_t);
extern template cudaError_t launch_tc_gemm_epi<EPI_GELU_AUX_BIAS>(int, int, int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                   const GemmArgs&, int, cudaStream_t);
extern template cudaError_t launch_tc_gemm_epi<EPI_DRELU_BGRAD>(int, int, int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                   const GemmArgs&, int, cudaStream_t);
extern template cudaError_t launch_tc_gemm_epi<EPI_DGELU_BGRAD>(int, int, int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                   const GemmArgs&, int, cudaStream_t);
extern template cudaError_t launch_tc_gemm_epi<EPI_BIAS_RESIDUAL>(int, int, int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                   const GemmArgs&, int, cudaStream_t);

namespace {

// Split-K fixup: warp items are (tail tile, row, 128-column group); lane l
// takes the four adjacent columns 4l..4l+3 of the group. The pieces' 16-byte
// loads are issued four at a time before they are added in piece order (the
// sum is the same as adding them one by one), then bias, activation, mask
// bits (a 32-column word gathered from the nibbles of 8 lanes) and the
// 16-bit stores. The grid is what fits on the GPU at once (64 registers a
// thread, 4 blocks per SM); warps stride over the items.
constexpr int kMaxSplit = 16;
constexpr int kFixupBlocksPerSm = 4;
__global__ void __launch_bounds__(256, kFixupBlocksPerSm) tc_gemm_fixup_kernel(const GemmArgs p, int tile_m, int bn) {
  grid_dependency_wait();  // the GEMM's pieces are complete and visible
  const int lane = threadIdx.x & 31;
  const int num_m = (p.Mk + tile_m - 1) / tile_m;
  const int num_n = (p.Nk + bn - 1) / bn;
  const int num_tiles = num_m * num_n;
  const int tail = num_tiles - p.tail_start;
  const int groups = bn / 128;
  const long long work = static_cast<long long>(tail) * tile_m * groups;
  const long long split_stride = static_cast<long long>(tile_m) * bn;
  const long long nw = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const bool bf16 = p.bf16 != 0;
  const unsigned short* bias16 = reinterpret_cast<const unsigned short*>(p.bias);
  unsigned short* D16 = reinterpret_cast<unsigned short*>(p.D);
  for (long long w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < work; w += nw) {
    const int t = static_cast<int>(w / (static_cast<long long>(tile_m) * groups));
    const int rem = static_cast<int>(w - static_cast<long long>(t) * tile_m * groups);
    const int r = rem / groups;
    const int g = rem - r * groups;
    int mt, nt;
    tile_coords(p.tail_start + t, num_m, num_n, p.group_m, mt, nt);
    const int grow = mt * tile_m + r;
    if (grow >= p.Mk) continue;
    const int gcol0 = nt * bn + g * 128 + 4 * lane;
    const float* src = p.partials + static_cast<long long>(t) * p.split * split_stride +
                       static_cast<long long>(r) * bn + g * 128 + 4 * lane;
    float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int s0 = 0; s0 < p.split; s0 += 4) {
      float4 pv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (s0 + i < p.split) pv[i] = __ldcg(reinterpret_cast<const float4*>(src + (s0 + i) * split_stride));
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (s0 + i < p.split) {
          z[0] += pv[i].x;
          z[1] += pv[i].y;
          z[2] += pv[i].z;
          z[3] += pv[i].w;
        }
    }
    unsigned short y16[4], z16[4];
    uint32_t nib = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int gcol = gcol0 + k;
      const bool in = gcol < p.Nk;
      if (p.epi != EPI_NONE && in) z[k] += to_f32(bf16, p.bias_per_col ? bias16[gcol] : bias16[grow]);
      y16[k] = from_f32(bf16, apply_act(p.epi, z[k]));
      z16[k] = from_f32(bf16, z[k]);
      if (in && z[k] > 0.0f) nib |= 1u << k;
    }
    const long long drow = static_cast<long long>(grow) * p.ldd;
    if (gcol0 + 3 < p.Nk) {  // (ldd is a multiple of 8 and gcol0 of 4: 8-byte aligned)
      *reinterpret_cast<uint2*>(D16 + drow + gcol0) =
          make_uint2(y16[0] | (static_cast<uint32_t>(y16[1]) << 16), y16[2] | (static_cast<uint32_t>(y16[3]) << 16));
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (gcol0 + k < p.Nk) D16[drow + gcol0 + k] = y16[k];
    }
    if (p.epi == EPI_GELU_AUX_BIAS) {
      const long long zrow = static_cast<long long>(grow) * p.ld_zaux;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (gcol0 + k < p.Nk) p.zaux[zrow + gcol0 + k] = z16[k];
    }
    if (p.epi == EPI_RELU_AUX_BIAS) {
      // the word of columns 32v..32v+31 of the group: lanes 8v..8v+7
      uint32_t word = nib << (4 * (lane & 7));
      word |= __shfl_xor_sync(0xffffffffu, word, 1);
      word |= __shfl_xor_sync(0xffffffffu, word, 2);
      word |= __shfl_xor_sync(0xffffffffu, word, 4);
      const int wcol0 = gcol0 - 4 * (lane & 7);  // first column of the word
      if ((lane & 7) == 0 && wcol0 < ((p.Nk + 127) & ~127))
        p.aux[static_cast<long long>(grow) * p.ld_aux + (wcol0 >> 5)] = word;
    }
  }
}

}  // namespace

cudaError_t launch_tc_gemm_fixup(int block_n, int pair, const GemmArgs& args, int num_sms, cudaStream_t stream) {
  const int tile_m = pair ? 2 * BM : BM;
  const long long num_tiles = static_cast<long long>((args.Mk + tile_m - 1) / tile_m) *
                              ((args.Nk + block_n - 1) / block_n);
  const long long warps = (num_tiles - args.tail_start) * tile_m * (block_n / 128);
  if (warps <= 0) return cudaSuccess;
  if (args.split > kMaxSplit) return cudaErrorInvalidValue;
  long long blocks = (warps + 7) / 8;
  const long long resident = static_cast<long long>(num_sms) * kFixupBlocksPerSm;
  if (blocks > resident) blocks = resident;
  // A programmatic dependent of the GEMM: it may be scheduled while the GEMM
  // runs and waits in the kernel for the GEMM's completion.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, tc_gemm_fixup_kernel, args, tile_m, block_n);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_tc_gemm(int block_n, int pair, int epi_warps, const CUtensorMap& tmA,
                           const CUtensorMap& tmB, const CUtensorMap& tmD, const CUtensorMap& tmZ,
                           const GemmArgs& args, int grid, cudaStream_t stream) {
  switch (args.epi) {
    case EPI_NONE: return launch_tc_gemm_epi<EPI_NONE>(block_n, pair, epi_warps, tmA, tmB, tmD, tmZ, args, grid, stream);
    case EPI_BIAS: return launch_tc_gemm_epi<EPI_BIAS>(block_n, pair, epi_warps, tmA, tmB, tmD, tmZ, args, grid, stream);
    case EPI_RELU_BIAS: return launch_tc_gemm_epi<EPI_RELU_BIAS>(block_n, pair, epi_warps, tmA, tmB, tmD, tmZ, args, grid, stream);
    case EPI_GELU_BIAS: return launch_tc_gemm_epi<EPI_GELU_BIAS>(block_n, pair, epi_warps, tmA, tmB, tmD, tmZ, args, grid, stream);
    case EPI_GELU_ERF_BIAS: return launch_tc_gemm_epi<EPI_GELU_ERF_BIAS>(block_n, pair, epi_warps, tmA, tmB, tmD, tmZ, args, grid, stream);
    case EPI_RELU_AUX_BIAS: return launch_tc_gemm_epi<EPI_RELU_AUX_BIAS>(block_n, pair, epi_warps, tmA, tmB, tmD, tmZ, args, grid, stream);
    case EPI_GELU_AUX_BIAS: return launch_tc_gemm_epi<EPI_GELU_AUX_BIAS>(block_n, pair, epi_warps, tmA, tmB, tmD, tmZ, args, grid, stream);
    case EPI_DRELU_BGRAD: return launch_tc_gemm_epi<EPI_DRELU_BGRAD>(block_n, pair, epi_warps, tmA, tmB, tmD, tmZ, args, grid, stream);
    case EPI_DGELU_BGRAD: return launch_tc_gemm_epi<EPI_DGELU_BGRAD>(block_n, pair, epi_warps, tmA, tmB, tmD, tmZ, args, grid, stream);
    case EPI_BIAS_RESIDUAL: return launch_tc_gemm_epi<EPI_BIAS_RESIDUAL>(block_n, pair, epi_warps, tmA, tmB, tmD, tmZ, args, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ge
