// ge_api.cu -- the C ABI (include/ge.h): argument validation, kernel-path
// choice, TMA tensor-map encoding and launches.
//
// The life cycle follows nvmath-python cuBLASLt bias-fusion guide, "Core API
// and parameter configuration" and "Advanced techniques" (plan once -- the
// expensive, blocking step that picks the kernel -- then execute many times,
// then free), and Fusing bias addition with matrix multiplication using
// nvmath-python (operands on one device with compatible dtypes, else an
// error; the plan must be freed).
#include <cudaTypedefs.h>

#include <array>
#include <cstdint>
#include <cstdlib>
#include <map>
#include <cstring>
#include <mutex>
#include <new>

#include "ge_internal.h"
#include "../../include/ge.h"

namespace {

using namespace ge;

constexpr long long kWaitBudgetCycles = 4000000000LL;  // ~2 s at GB300 clocks

struct Plan {
  int64_t M = 0, N = 0, K = 0;
  ge_epilogue_t epi = GE_EPI_NONE;
  ge_layout_t L{};
  ge_path_t path = GE_PATH_TC_GEMM;
  int device = 0;
  int num_sms = 0;
  // tensor-core path: kernel-level problem after folding a column-major D
  bool swap = false;
  int block_n = 256;
  int pair = 0;  // 2-CTA (cta_group::2) tiles of 256 rows
  int epi_warps = 4;  // epilogue warps of the tensor-core kernel (4 or 8)
  int kb = 64;        // k-values per pipeline stage (64 or 128)
  int tail_start = 0;  // split-K tail (see GemmArgs); `tail_ws` holds its pieces
  int split = 1;
  int sk_tiles = 0;    // stream-K tiles (see GemmArgs); `tail_ws` holds the workers' slots
  unsigned int* sk_sync = nullptr;  // stream-K epoch, counter and flags (in `ws`)
  bool chain_ok = false;            // ge_execute_chain accepts the plan (see the path choice)
  unsigned int* chain_x = nullptr;  // ge_execute_chain's exchange words (in `ws`)
  int chain_producers = 0, chain_inflight = 0;  // ge_execute_chain tuning (0: defaults)
  int two_producers = -1;           // tensor-core GEMM: a second producer warp issues B (-1: by layout)
  void* tail_ws = nullptr;  // separate allocation (re-sized by autotune)
  size_t tail_ws_bytes = 0;
  bool tc_allow_split = true;
  float2* nstats = nullptr;    // norm plans, tensor-core path: per (n-tile, token) statistics
  float2* rowstats = nullptr;  // ... and per token (mean, rstd)
  float* bg_partials = nullptr;  // DRELU_BGRAD GEMM epilogue: bias-gradient partials
  long long bg_rows = 0, bg_len = 0;
  int grid = 0;
  int group_m = 16;
  // stored D: R rows x C contiguous
  int64_t R = 0, C = 0;
  int64_t aux_words = 0;  // ld_aux: mask words, or elements of the 16-bit z (GELU_AUX / DGELU)
  int static_a = 0;       // GE_ATTR_STATIC_A
  int bf16 = 0;           // element type of A, B, D and bias: 0 fp16, 1 bf16
  // device workspace: [error word | pad to 256 | counters | partials]
  void* ws = nullptr;
  size_t ws_bytes = 0;
  unsigned int* err = nullptr;
  unsigned int* counters = nullptr;
  float* partials = nullptr;
  int splits = 1;
  // tensor-map cache (rebuilt when a pointer changes)
  const void* mapA = nullptr;
  const void* mapB = nullptr;
  const void* mapD = nullptr;
  const void* mapZ = nullptr;
  CUtensorMap tmA{}, tmB{}, tmD{}, tmZ{};
  // last pointers whose device was verified, and the driver's id of the
  // allocation each one was in at the time
  const void* checked[6] = {};
  unsigned long long checked_id[6] = {};
  // ge_execute_chain: the weight and bias pointers verified so far, with
  // their allocations' ids
  std::map<const void*, unsigned long long> chain_checked;
  // DW_DRELU_BGRAD run as two launches (the default): the standalone
  // DRELU_BGRAD pass into dz_ws ([K][lda] elements), then the NONE GEMM on
  // it; bg_scratch takes the bias gradient when the caller wants none.
  Plan* sub_drelu = nullptr;
  Plan* sub_gemm = nullptr;
  void* dz_ws = nullptr;
  float* bg_scratch = nullptr;
};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D tensor map of 16-bit elements (fp16, or bf16 when `bf16`): inner extent
// d0 (contiguous), outer d1, row pitch ld elements, box b0 x b1, swizzle mode.
bool make_map(CUtensorMap* m, int bf16, const void* base, uint64_t d0, uint64_t d1, uint64_t ld,
              uint32_t b0, uint32_t b1, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {d0, d1};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {b0, b1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// K-major 16-bit operand of `rows` rows with K = 64 * panels contiguous
// elements (row pitch ld) seen as 3-D: 64 elements x rows x panels, so that
// one box (64 x box_rows x box_panels, 128-byte swizzle) fetches several
// 64-wide panels at once. Only for K a multiple of 64: a panel never runs
// past the end of a row.
bool make_map_panels(CUtensorMap* m, int bf16, const void* base, uint64_t rows, uint64_t panels, uint64_t ld,
                     uint32_t box_rows, uint32_t box_panels) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, rows, panels};
  cuuint64_t strides[2] = {ld * 2, 128};
  cuuint32_t box[3] = {64, box_rows, box_panels};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base),
                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool epi_is_norm(ge_epilogue_t e) {
  return e == GE_EPI_BIAS_RESIDUAL_RMSNORM || e == GE_EPI_BIAS_RESIDUAL_LAYERNORM;
}

bool epi_has_bias(ge_epilogue_t e) {
  return e == GE_EPI_BIAS || e == GE_EPI_RELU_BIAS || e == GE_EPI_GELU_BIAS ||
         e == GE_EPI_RELU_AUX_BIAS || e == GE_EPI_GELU_ERF_BIAS || e == GE_EPI_GELU_AUX_BIAS;
}

// The driver's unique id of the allocation holding `p` (0 if unknown): a
// pointer value freed and handed out again, possibly on another device of
// the same address space, gets a new id.
using PFN_pointerGetAttribute = CUresult (*)(void*, CUpointer_attribute, CUdeviceptr);
unsigned long long buffer_id(const void* p) {
  static PFN_pointerGetAttribute fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_pointerGetAttribute>(f);
  });
  unsigned long long id = 0;
  if (!fn || fn(&id, CU_POINTER_ATTRIBUTE_BUFFER_ID, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS) {
    cudaGetLastError();
    return 0;
  }
  return id;
}

// Verify that `p` is device memory of the plan's device. The result is
// cached per slot for the same pointer in the same allocation; a pointer
// whose allocation changed (freed and reallocated) is verified again.
ge_status_t check_device(Plan* pl, int slot, const void* p) {
  if (!p) return GE_OK;
  const unsigned long long id = buffer_id(p);
  if (pl->checked[slot] == p && id != 0 && pl->checked_id[slot] == id) return GE_OK;
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GE_ERR_DEVICE_MISMATCH;
  }
  if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
    return GE_ERR_DEVICE_MISMATCH;
  if (at.device != pl->device) return GE_ERR_DEVICE_MISMATCH;
  pl->checked[slot] = p;
  pl->checked_id[slot] = id;
  return GE_OK;
}

// Tensor-core launch configuration for a tile width and pair mode: work
// units, grid, rasterisation group and the split-K tail.
struct TcConfig {
  int block_n = 256, pair = 0, split = 1, tail_start = 0, grid = 1, group_m = 1, kb = 64, sk_tiles = 0;
};

// k-values per pipeline stage for a tile shape: 128 (two 64-wide panels per
// operand box) when K is a multiple of 128 and a stage stays within 64 KB
// (2-SM pairs, or 128-wide single-CTA tiles); 64 otherwise, and always for
// the masked-operand weight gradient. GE_KB = 64 forces one panel (sweeps).
// (Four panels, 96 KB stages, on 256 x 128 pair tiles measured slower:
// 4096 x 512 x 4096 GELU_BIAS 26.8 vs 25.5 us.)
int kb_for(const Plan& pl, int block_n, int pair) {
  const bool fits = pl.K % 128 == 0 && (pair || block_n == 128) && pl.epi != GE_EPI_DW_DRELU_BGRAD;
  if (const char* env = std::getenv("GE_KB"))
    if (env[0] == '6') return 64;
  return fits ? 128 : 64;
}

// Configurations chosen by ge_plan_autotune, per device, problem and layout:
// a plan created later for the same key starts from the tuned choice.
struct TunedChoice {
  int block_n, pair, split, sk, kb;
};
using TuneKey = std::array<int64_t, 13>;
std::map<TuneKey, TunedChoice>& tuned_cache() {
  static std::map<TuneKey, TunedChoice> m;
  return m;
}
std::mutex& tuned_mutex() {
  static std::mutex mu;
  return mu;
}
TuneKey tune_key(const Plan& pl) {
  return {pl.device, pl.M, pl.N, pl.K, static_cast<int64_t>(pl.epi), pl.bf16, pl.L.a, pl.L.b, pl.L.d,
          pl.L.lda, pl.L.ldb, pl.L.ldd, pl.L.ld_aux};
}

// kb64: stages of one 64-wide k panel even where two would fit (an autotune
// candidate).
TcConfig tc_config(const Plan& pl, int block_n, int pair, bool allow_split, bool kb64 = false) {
  if (block_n == 224) allow_split = false;  // the fixup reads 128-column groups
  TcConfig c;
  c.block_n = block_n;
  c.pair = pair;
  c.kb = kb64 ? 64 : kb_for(pl, block_n, pair);
  const int64_t Mk = pl.swap ? pl.N : pl.M;
  const int64_t Nk = pl.swap ? pl.M : pl.N;
  const int64_t tile_m = pair ? 256 : 128;
  const long long num_m = (Mk + tile_m - 1) / tile_m;
  const long long num_n = (Nk + block_n - 1) / block_n;
  const long long tiles = num_m * num_n;
  const long long workers = pair ? tc_gemm_max_pairs(block_n, pl.num_sms, pl.epi_warps) : pl.num_sms;
  // Tiles go out in groups of 16 m-tiles sweeping the n-tiles, so that the
  // group's A rows are reused from L2 (2-SM pairs, 11008x8192x4096 forward:
  // 16 rows 0.4205 ms, 8 rows 0.4315; the whole 32-row panel 0.440 ms and
  // twice the DRAM reads, its A re-read once the 180 MB output has streamed
  // through L2).
  c.group_m = static_cast<int>(num_m < 16 ? num_m : 16);
  if (const char* env = std::getenv("GE_GROUP_M")) {  // rasterisation sweeps
    const long long g = std::atoll(env);
    if (g >= 1) c.group_m = static_cast<int>(g < num_m ? g : num_m);
  }
  // Split-K tail: when the last of several waves would leave most workers
  // idle, the tiles of that wave are split along K into just enough pieces
  // to occupy the workers (at least 4 k-blocks per piece, at most 16); a
  // fixup kernel adds the fp32 pieces in order and applies the epilogue.
  // (Measured: dW 11008x4096x8192 0.423 -> 0.397 ms.) A problem whose only
  // wave leaves at least half of the workers idle is split whole the same
  // way: the fixup is launched as a programmatic dependent of the GEMM, so
  // its launch overlaps the GEMM (1024x512x2048 GELU_BIAS, 32 tiles: 25.0 ->
  // 21.9 us; 4096x128x4096: 34.0 -> 25.5 us).
  // Stream-K (GE_STREAM_K = 1, for any ragged last wave): the last one or
  // two waves' tiles are shared out as equal ranges of k-block iterations
  // (each tile then in about W / sk_tiles + 1 pieces) and every tile is
  // finished inside the GEMM by the worker that starts it. Not the default:
  // measured slower than the plain waves on the shapes it is for (FFN up
  // 4096x2048x4096: 73 vs 58 us; 4096x512x4096: 36 vs 30 us), because the
  // finisher's epilogue (a whole tile's, plus adding the pieces) lands at
  // the very end of every worker's range.
  const long long num_kb = (pl.K + c.kb - 1) / c.kb;
  const long long rem = tiles % workers;
  auto pieces = [&](long long t) {
    long long S = workers / t;
    if (S > num_kb / 4) S = num_kb / 4;
    return S > 16 ? 16LL : S;
  };
  int sk_env = -1;
  if (const char* env = std::getenv("GE_STREAM_K")) sk_env = env[0] == '0' ? 0 : (env[0] == '1' ? 1 : -1);
  // (not for the masked-operand weight gradient: its bias-gradient partials
  // are per split-K piece)
  const bool sk_ok = allow_split && rem != 0 && sk_env != 0 && pl.epi != GE_EPI_DW_DRELU_BGRAD;
  if (sk_ok && sk_env == 1) {
    c.sk_tiles = static_cast<int>(tiles < 2 * workers ? tiles : rem + workers);
  } else if (allow_split && tiles > workers && rem != 0 && rem * 2 <= workers) {
    const long long S = pieces(rem);
    if (S >= 2) {
      c.split = static_cast<int>(S);
      c.tail_start = static_cast<int>(tiles - rem);
    }
  } else if (allow_split && tiles * 2 <= workers) {
    const long long S = pieces(tiles);
    if (S >= 2) {
      c.split = static_cast<int>(S);
      c.tail_start = 0;
    }
  }
  if (c.split == 1) c.tail_start = static_cast<int>(tiles);
  if (c.sk_tiles > 0) {
    c.grid = static_cast<int>(pair ? 2 * workers : workers);  // every worker has a range
  } else {
    const long long units = c.tail_start + (tiles - c.tail_start) * c.split;
    const long long g = units < workers ? units : workers;
    c.grid = static_cast<int>(pair ? 2 * g : g);
  }
  return c;
}

size_t tc_tail_bytes(const Plan& pl, const TcConfig& c) {
  if (c.sk_tiles > 0) {  // one slot per worker
    const int64_t tile_m = c.pair ? 256 : 128;
    const int64_t workers = c.pair ? c.grid / 2 : c.grid;
    return static_cast<size_t>(workers) * tile_m * c.block_n * 4;
  }
  if (c.split <= 1) return 0;
  const int64_t Mk = pl.swap ? pl.N : pl.M;
  const int64_t Nk = pl.swap ? pl.M : pl.N;
  const int64_t tile_m = c.pair ? 256 : 128;
  const int64_t tiles = ((Mk + tile_m - 1) / tile_m) * ((Nk + c.block_n - 1) / c.block_n);
  return static_cast<size_t>(tiles - c.tail_start) * c.split * tile_m * c.block_n * 4;
}

// Make `c` the plan's configuration (re-sizing the tail workspace).
ge_status_t apply_config(Plan* pl, const TcConfig& c) {
  const size_t need = tc_tail_bytes(*pl, c);
  if (need > pl->tail_ws_bytes) {
    void* p = nullptr;
    if (cudaMalloc(&p, need) != cudaSuccess) {
      cudaGetLastError();
      return GE_ERR_OOM;
    }
    if (pl->tail_ws) cudaFree(pl->tail_ws);
    pl->tail_ws = p;
    pl->tail_ws_bytes = need;
  }
  pl->block_n = c.block_n;
  pl->pair = c.pair;
  pl->kb = c.kb;
  pl->split = c.split;
  pl->tail_start = c.tail_start;
  pl->sk_tiles = c.sk_tiles;
  pl->grid = c.grid;
  pl->group_m = c.group_m;
  pl->partials = static_cast<float*>(pl->tail_ws);
  pl->mapA = pl->mapB = pl->mapD = pl->mapZ = nullptr;  // B's box depends on the pair mode
  return GE_OK;
}

// Tensor maps for the tensor-core path (kernel-level operands A', B', D' and,
// for GELU_AUX_BIAS, the z output Z' stored like D'; otherwise tmZ repeats
// D's map and is not used).
// Mask words (DW_DRELU_BGRAD): rows of ld_aux uint32 words, K rows; a box of
// 4 words (128 m) x 64 k-rows, no swizzle.
bool make_mask_map(CUtensorMap* m, const void* base, uint64_t words, uint64_t rows, uint64_t ld_words) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {words, rows};
  cuuint64_t strides[1] = {ld_words * 4};
  cuuint32_t box[2] = {4, 64};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

ge_status_t build_maps(Plan* pl, const void* A, const void* B, void* D, void* Z) {
  if (!Z) Z = D;
  if (pl->mapA == A && pl->mapB == B && pl->mapD == D && pl->mapZ == Z) return GE_OK;
  const ge_layout_t& L = pl->L;
  const void* Ak = pl->swap ? B : A;
  const void* Bk = pl->swap ? A : B;
  const int a_mn = pl->swap ? (L.b == GE_MN_MAJOR) : (L.a == GE_MN_MAJOR);
  const int b_mn = pl->swap ? (L.a == GE_MN_MAJOR) : (L.b == GE_MN_MAJOR);
  const int64_t lda = pl->swap ? L.ldb : L.lda;
  const int64_t ldb = pl->swap ? L.lda : L.ldb;
  const uint64_t Mk = pl->swap ? pl->N : pl->M;
  const uint64_t Nk = pl->swap ? pl->M : pl->N;
  const uint64_t K = pl->K;
  bool ok = true;
  const uint32_t b_rows = static_cast<uint32_t>(pl->pair ? pl->block_n / 2 : pl->block_n);
  const uint32_t kb = static_cast<uint32_t>(pl->kb);
  if (!a_mn)
    ok &= kb >= 128 ? make_map_panels(&pl->tmA, pl->bf16, Ak, Mk, K / 64, lda, 128, kb / 64)
                    : make_map(&pl->tmA, pl->bf16, Ak, K, Mk, lda, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  else
    ok &= make_map(&pl->tmA, pl->bf16, Ak, Mk, K, lda, 64, kb, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!b_mn)
    ok &= kb >= 128 ? make_map_panels(&pl->tmB, pl->bf16, Bk, Nk, K / 64, ldb, b_rows, kb / 64)
                    : make_map(&pl->tmB, pl->bf16, Bk, K, Nk, ldb, 64, b_rows, CU_TENSOR_MAP_SWIZZLE_128B);
  else
    ok &= make_map(&pl->tmB, pl->bf16, Bk, Nk, K, ldb, 64, kb, CU_TENSOR_MAP_SWIZZLE_128B);
  ok &= make_map(&pl->tmD, pl->bf16, D, Nk, Mk, L.ldd, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
  if (pl->epi == GE_EPI_DW_DRELU_BGRAD)  // the fourth map carries the mask words
    ok &= make_mask_map(&pl->tmZ, Z, static_cast<uint64_t>(L.ld_aux), K, static_cast<uint64_t>(L.ld_aux));
  else
    ok &= make_map(&pl->tmZ, pl->bf16, Z, Nk, Mk, Z == D ? L.ldd : L.ld_aux, 32, 32,
                   CU_TENSOR_MAP_SWIZZLE_64B);
  if (!ok) {
    pl->mapA = pl->mapB = pl->mapD = pl->mapZ = nullptr;
    return GE_ERR_CUDA;
  }
  pl->mapA = A;
  pl->mapB = B;
  pl->mapD = D;
  pl->mapZ = Z;
  return GE_OK;
}

ge_status_t launch_forward(Plan* pl, const void* A, const void* B, const void* bias, void* D,
                           void* aux, int epi_code, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  if (pl->path == GE_PATH_GEMV) {
    GemvArgs g{};
    g.M = static_cast<int>(pl->M);
    g.N = static_cast<int>(pl->N);
    g.K = static_cast<int>(pl->K);
    g.A = static_cast<const __half*>(A);
    g.lda = pl->L.lda;
    g.B = static_cast<const __half*>(B);
    g.ldb = pl->L.ldb;
    g.D = static_cast<__half*>(D);
    g.ldd_m = pl->L.d == GE_D_ROW ? pl->L.ldd : 1;
    g.ldd_n = pl->L.d == GE_D_ROW ? 1 : pl->L.ldd;
    g.bias = static_cast<const __half*>(bias);
    g.res = epi_code == EPI_BIAS_RESIDUAL ? static_cast<const unsigned short*>(aux) : nullptr;
    g.epi = epi_code;
    g.static_a = pl->static_a;
    g.bf16 = pl->bf16;
    g.err = pl->err;
    e = launch_gemv(g, pl->num_sms, st);
  } else {
    const bool zout = epi_code == EPI_GELU_AUX_BIAS;
    const bool mask_map = pl->epi == GE_EPI_DW_DRELU_BGRAD;
    ge_status_t s = build_maps(pl, A, B, D, (zout || mask_map) ? aux : nullptr);
    if (s != GE_OK) return s;
    GemmArgs g{};
    g.Mk = static_cast<int>(pl->swap ? pl->N : pl->M);
    g.Nk = static_cast<int>(pl->swap ? pl->M : pl->N);
    g.K = static_cast<int>(pl->K);
    g.a_mn = pl->swap ? (pl->L.b == GE_MN_MAJOR) : (pl->L.a == GE_MN_MAJOR);
    g.b_mn = pl->swap ? (pl->L.a == GE_MN_MAJOR) : (pl->L.b == GE_MN_MAJOR);
    g.epi = epi_code;
    g.bias_per_col = pl->swap ? 1 : 0;
    g.bias = static_cast<const __half*>(bias);
    const bool zaux = epi_code == EPI_GELU_AUX_BIAS || epi_code == EPI_DGELU_BGRAD ||
                      epi_code == EPI_BIAS_RESIDUAL;
    g.aux = zaux ? nullptr : static_cast<uint32_t*>(aux);
    g.ld_aux = pl->aux_words;
    g.zaux = zaux ? static_cast<unsigned short*>(aux) : nullptr;
    g.ld_zaux = pl->aux_words;
    g.D = static_cast<__half*>(D);
    g.ldd = pl->L.ldd;
    g.err = pl->err;
    g.group_m = pl->group_m;
    // a second producer warp issues B when an operand is M/N-major (its
    // stage is then three or four TMA boxes, more than one thread issues in
    // step with the MMAs: dW 11008x4096x8192 365 -> 356 us); K-major stages
    // are two boxes and gain nothing (GE_TWO_PRODUCERS = 0 | 1 overrides)
    g.two_producers = pl->two_producers >= 0 ? pl->two_producers : (g.a_mn || g.b_mn ? 1 : 0);
    g.budget = kWaitBudgetCycles;
    g.tail_start = pl->tail_start;
    g.split = pl->split;
    g.partials = pl->partials;
    g.sk_tiles = pl->sk_tiles;
    g.sk_sync = pl->sk_sync;
    g.bg_partials = pl->bg_partials;
    g.bf16 = pl->bf16;
    g.nstats = epi_code == EPI_BIAS_RESIDUAL ? pl->nstats : nullptr;
    g.kb = pl->kb;
    const bool backward = epi_code == EPI_DRELU_BGRAD || epi_code == EPI_DGELU_BGRAD;
    g.bgrad = backward ? static_cast<float*>(const_cast<void*>(bias)) : nullptr;
    if (backward) g.bias = nullptr;
    const bool amask = pl->epi == GE_EPI_DW_DRELU_BGRAD;
    if (amask) {  // D = (A masked) . B, no epilogue arithmetic; bgrad from the transform warps
      g.epi = EPI_NONE;
      g.amask = 1;
      g.bias = nullptr;
      g.aux = nullptr;
      g.bgrad = static_cast<float*>(const_cast<void*>(bias));
      g.bg_partials = g.bgrad ? pl->bg_partials : nullptr;
    }
    e = launch_tc_gemm(pl->block_n, pl->pair, pl->epi_warps, pl->tmA, pl->tmB, pl->tmD, pl->tmZ, g, pl->grid, st);
    if (e == cudaSuccess && pl->split > 1) e = launch_tc_gemm_fixup(pl->block_n, pl->pair, g, pl->num_sms, st);
    if (e == cudaSuccess && amask && g.bgrad)
      e = launch_bgrad_reduce(pl->bg_partials, pl->split > 1 ? pl->split : 1, g.Mk, g.bgrad, st);
    if (e == cudaSuccess && backward) {
      const long long rows =
          pl->swap ? pl->bg_rows : (pl->epi_warps / 4) * static_cast<long long>((g.Nk + pl->block_n - 1) / pl->block_n);
      e = launch_bgrad_reduce(pl->bg_partials, rows, pl->bg_len, g.bgrad, st);
    }
  }
  return e == cudaSuccess ? GE_OK : GE_ERR_CUDA;
}

// Checks shared by the fused and unfused norm entry points.
ge_status_t check_norm_args(Plan* pl, const void* A, const void* B, const void* bias, const void* residual,
                            const void* gamma, const void* beta, const void* H, const void* Y) {
  if (!pl) return GE_ERR_INVALID_ARG;
  if (!epi_is_norm(pl->epi)) return GE_ERR_UNSUPPORTED;
  const bool layer = pl->epi == GE_EPI_BIAS_RESIDUAL_LAYERNORM;
  if (!A || !B || !bias || !residual || !gamma || !H || !Y || (layer && !beta)) return GE_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(H) || !aligned16(Y) || !aligned16(residual) ||
      !aligned16(gamma) || (layer && !aligned16(beta)) || (reinterpret_cast<uintptr_t>(bias) & 1u))
    return GE_ERR_ALIGNMENT;
  ge_status_t s;
  if ((s = check_device(pl, 0, A)) != GE_OK || (s = check_device(pl, 1, B)) != GE_OK ||
      (s = check_device(pl, 2, bias)) != GE_OK || (s = check_device(pl, 3, H)) != GE_OK ||
      (s = check_device(pl, 4, residual)) != GE_OK || (s = check_device(pl, 5, Y)) != GE_OK)
    return s;
  return GE_OK;
}

// stats_ready: the GEMM epilogue has written the per-tile statistics.
ge_status_t launch_norm_pass(Plan* pl, const void* gamma, const void* beta, const void* H, void* Y, float eps,
                             bool stats_ready, cudaStream_t st) {
  NormArgs n{};
  n.R = pl->N;  // tokens: rows of the column-major D
  n.C = pl->M;  // features
  n.ld = pl->L.ldd;
  n.H = static_cast<const unsigned short*>(H);
  n.Y = static_cast<unsigned short*>(Y);
  n.gamma = static_cast<const unsigned short*>(gamma);
  n.beta = static_cast<const unsigned short*>(beta);
  n.eps = eps;
  n.layer = pl->epi == GE_EPI_BIAS_RESIDUAL_LAYERNORM ? 1 : 0;
  n.bf16 = pl->bf16;
  if (stats_ready && pl->nstats) {
    n.partials = pl->nstats;
    n.tile_w = pl->block_n;
    n.ntiles = static_cast<int>((pl->M + pl->block_n - 1) / pl->block_n);
    n.halves = pl->epi_warps / 4;
    n.rowstats = pl->rowstats;
  }
  return launch_norm(n, pl->num_sms, st) == cudaSuccess ? GE_OK : GE_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* ge_version(void) { return "0.1.0"; }

const char* ge_status_string(ge_status_t s) {
  switch (s) {
    case GE_OK: return "GE_OK";
    case GE_ERR_INVALID_ARG: return "GE_ERR_INVALID_ARG: invalid argument";
    case GE_ERR_UNSUPPORTED: return "GE_ERR_UNSUPPORTED: dtype/epilogue/layout not supported";
    case GE_ERR_ALIGNMENT: return "GE_ERR_ALIGNMENT: pointer or leading dimension not 16-byte aligned";
    case GE_ERR_DEVICE_MISMATCH: return "GE_ERR_DEVICE_MISMATCH: buffer not on the plan's device";
    case GE_ERR_CUDA: return "GE_ERR_CUDA: CUDA call or launch failed";
    case GE_ERR_TIMEOUT: return "GE_ERR_TIMEOUT: a bounded device wait expired";
    case GE_ERR_OOM: return "GE_ERR_OOM: workspace allocation failed";
    case GE_ERR_DEVICE_CHECK: return "GE_ERR_DEVICE_CHECK: a device-side index or phase check failed (debug build)";
  }
  return "unknown ge_status_t";
}

ge_status_t ge_plan_create(ge_plan_t* out, int64_t M, int64_t N, int64_t K, ge_dtype_t a,
                           ge_dtype_t b, ge_dtype_t d, ge_dtype_t compute, ge_epilogue_t epi,
                           const ge_layout_t* layout) {
  if (!out) return GE_ERR_INVALID_ARG;
  *out = nullptr;
  if (static_cast<int>(epi) < GE_EPI_NONE || static_cast<int>(epi) > GE_EPI_DW_DRELU_BGRAD)
    return GE_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 0) return GE_ERR_INVALID_ARG;
  const int64_t lim = (int64_t(1) << 31) - 1;
  if (M > lim || N > lim || K > lim) return GE_ERR_INVALID_ARG;
  // A, B, D (and the bias) share one 16-bit element type; products are
  // accumulated in fp32 either way.
  if (a != b || a != d || (a != GE_F16 && a != GE_BF16) || compute != GE_F32) return GE_ERR_UNSUPPORTED;
  const bool backward = epi == GE_EPI_DRELU_BGRAD || epi == GE_EPI_DGELU_BGRAD;
  if (!backward && K == 0) return GE_ERR_INVALID_ARG;
  ge_layout_t L{GE_K_MAJOR, GE_MN_MAJOR, GE_D_ROW, 0, 0, 0, 0};
  if (layout) L = *layout;
  if ((L.a != GE_K_MAJOR && L.a != GE_MN_MAJOR) || (L.b != GE_K_MAJOR && L.b != GE_MN_MAJOR) ||
      (L.d != GE_D_ROW && L.d != GE_D_COL))
    return GE_ERR_INVALID_ARG;
  if (L.lda < 0 || L.ldb < 0 || L.ldd < 0 || L.ld_aux < 0) return GE_ERR_INVALID_ARG;
  // The norm runs over the M features of each token: they must be the
  // contiguous index of D (D column-major, i.e. Y[N tokens][M features]).
  if (epi_is_norm(epi) && L.d != GE_D_COL) return GE_ERR_UNSUPPORTED;
  // The masked-operand weight gradient: A = dY read M-major ([K tokens][M]),
  // its mask packed along M per token, D row-major (the kernel's own A').
  const bool dw_mask = epi == GE_EPI_DW_DRELU_BGRAD;
  if (dw_mask && (L.a != GE_MN_MAJOR || L.d != GE_D_ROW)) return GE_ERR_UNSUPPORTED;

  Plan tmp;
  tmp.M = M;
  tmp.N = N;
  tmp.K = K;
  tmp.epi = epi;
  tmp.bf16 = a == GE_BF16 ? 1 : 0;
  tmp.R = L.d == GE_D_ROW ? M : N;
  tmp.C = L.d == GE_D_ROW ? N : M;

  // A 1-column B (decode) stored N-major with unit pitch is a contiguous
  // vector, the same bytes as K-major: read it as K-major.
  const bool standalone_drelu = backward && K == 0;
  if (!standalone_drelu && N == 1 && L.b == GE_MN_MAJOR && (L.ldb == 0 || L.ldb == 1)) {
    L.b = GE_K_MAJOR;
    L.ldb = (K + 7) / 8 * 8;
  }
  if (!standalone_drelu) {
    const int64_t min_lda = L.a == GE_K_MAJOR ? K : M;
    const int64_t min_ldb = L.b == GE_K_MAJOR ? K : N;
    if (L.lda == 0) L.lda = min_lda;
    if (L.ldb == 0) L.ldb = min_ldb;
    if (L.lda < min_lda || L.ldb < min_ldb) return GE_ERR_INVALID_ARG;
  }
  if (L.ldd == 0) L.ldd = tmp.C;
  if (L.ldd < tmp.C) return GE_ERR_INVALID_ARG;
  const bool has_mask = epi == GE_EPI_RELU_AUX_BIAS || epi == GE_EPI_DRELU_BGRAD;
  if (has_mask) {
    const int64_t min_words = (tmp.C + 31) / 32;
    if (L.ld_aux == 0) L.ld_aux = (tmp.C + 127) / 128 * 4;
    if (L.ld_aux < min_words) return GE_ERR_INVALID_ARG;
    if (L.ld_aux % 4 != 0) return GE_ERR_ALIGNMENT;
    tmp.aux_words = L.ld_aux;
  }
  if (dw_mask) {  // mask rows are the K tokens, words along the M features
    if (L.ld_aux == 0) L.ld_aux = (M + 127) / 128 * 4;
    if (L.ld_aux < (M + 31) / 32) return GE_ERR_INVALID_ARG;
    if (L.ld_aux % 4 != 0) return GE_ERR_ALIGNMENT;
    tmp.aux_words = L.ld_aux;
  }
  const bool has_zaux = epi == GE_EPI_GELU_AUX_BIAS || epi == GE_EPI_DGELU_BGRAD;
  if (epi_is_norm(epi)) tmp.aux_words = L.ldd;  // residual, H and Y share D's layout
  if (has_zaux) {  // 16-bit z stored like D: ld_aux in elements, 16-byte rows
    if (L.ld_aux == 0) L.ld_aux = (tmp.C + 7) / 8 * 8;
    if (L.ld_aux < tmp.C) return GE_ERR_INVALID_ARG;
    if (L.ld_aux % 8 != 0) return GE_ERR_ALIGNMENT;
    tmp.aux_words = L.ld_aux;
  }

  // Path choice. Up to 16 tokens with K-major operands and no mask, aux or
  // backward output fit the weight-streaming GEMV; from 5 tokens on, with a
  // plain epilogue and D's stride a multiple of 8, the tensor-core kernel is
  // faster (its one wave split along K; 4096 x N x 4096 GELU_BIAS: N = 4
  // 25.3 us either way, N = 8 25.7 against 33.4 us for the GEMV, N = 16 22.1
  // against 84.6; 11008 x 16 x 4096: 29.3 against 160.4), the GEMV's
  // CUDA-core dot products being its bound as the tokens grow.
  const bool gemv_shape = !standalone_drelu && N <= 16 && L.a == GE_K_MAJOR && L.b == GE_K_MAJOR &&
                          epi != GE_EPI_RELU_AUX_BIAS && !has_zaux && !backward && !dw_mask;
  const bool few_tokens_tc = N >= 5 && (epi == GE_EPI_NONE || epi == GE_EPI_BIAS || epi == GE_EPI_RELU_BIAS ||
                                        epi == GE_EPI_GELU_BIAS || epi == GE_EPI_GELU_ERF_BIAS);
  // A plan a decode stack (ge_execute_chain) can run on, whichever kernel
  // its own execute takes: square, D column-major, no norm.
  tmp.chain_ok = gemv_shape && M == K && L.d == GE_D_COL && !epi_is_norm(epi);
  if (standalone_drelu) {
    tmp.path = GE_PATH_DRELU;
    if (L.ldd % 8 != 0) return GE_ERR_ALIGNMENT;
  } else if (gemv_shape && !(few_tokens_tc && L.ldd % 8 == 0)) {
    tmp.path = GE_PATH_GEMV;
    if (L.lda % 8 != 0 || L.ldb % 8 != 0) return GE_ERR_ALIGNMENT;
  } else {
    tmp.path = GE_PATH_TC_GEMM;
    if (L.lda % 8 != 0 || L.ldb % 8 != 0 || L.ldd % 8 != 0) return GE_ERR_ALIGNMENT;
  }
  tmp.L = L;

  // Device resources (the only CUDA calls of planning).
  if (cudaGetDevice(&tmp.device) != cudaSuccess) {
    cudaGetLastError();
    return GE_ERR_CUDA;
  }
  if (cudaDeviceGetAttribute(&tmp.num_sms, cudaDevAttrMultiProcessorCount, tmp.device) !=
      cudaSuccess) {
    cudaGetLastError();
    return GE_ERR_CUDA;
  }
  int tc_block_n = 256, tc_pair = 0;
  bool tc_split = true;
  if (tmp.path == GE_PATH_TC_GEMM) {
    tmp.swap = L.d == GE_D_COL;
    const int64_t Mk = tmp.swap ? N : M;
    const int64_t Nk = tmp.swap ? M : N;
    const long long t256 = ((Mk + 127) / 128) * ((Nk + 255) / 256);
    // 128 x 256 tiles move a third less shared-memory traffic per flop than
    // 128 x 128 ones (measured: the 11008x4096x8192 dW GEMM runs 1.54x faster
    // with them), so 128-wide tiles are used only when 256-wide ones would
    // leave more than half of the SMs without a tile.
    tc_block_n = (Nk <= 128 || t256 * 2 < tmp.num_sms) ? 128 : 256;
    int want_n = 0;
    if (const char* env = std::getenv("GE_TILE_N")) {  // tile-width sweeps
      want_n = std::atoi(env);
      if (want_n == 128 || want_n == 256) tc_block_n = want_n;
      if (want_n == 224) tc_block_n = 256;  // (narrowed below when the layout allows)
    }
    // 2-CTA pairs (256-row tiles) once there are enough of them to give
    // every pair of SMs at least one tile.
    const long long pair_tiles = ((Mk + 255) / 256) * ((Nk + tc_block_n - 1) / tc_block_n);
    tc_pair = (tc_block_n == 256 && pair_tiles * 2 >= tmp.num_sms) ? 1 : 0;
    if (const char* env = std::getenv("GE_PAIR")) {
      if (env[0] == '0') tc_pair = 0;
      if (env[0] == '1') tc_pair = 1;
    }
    // 256 x 224 pair tiles when 256-wide ones end in a last wave too full
    // for the split-K tail and the narrower tiles make the waves come out
    // shorter: e.g. 4096 x 2048 x 4096 (D column-major): 128 tiles of 256 x
    // 256 on 76 pairs (two waves, the second 68 % full) or 152 of 256 x 224
    // (two full waves of tiles an eighth shorter). K-major B' only (its 112
    // rows a CTA are staged in 128-byte swizzle rows), no split-K tail.
    const bool bmn_k = tmp.swap ? (L.a == GE_MN_MAJOR) : (L.b == GE_MN_MAJOR);
    if (tc_pair && tc_block_n == 256 && !bmn_k && !dw_mask) {
      const long long W = tmp.num_sms / 2;
      const long long m_t = (Mk + 255) / 256;
      const long long t256p = m_t * ((Nk + 255) / 256), t224p = m_t * ((Nk + 223) / 224);
      const long long rem = t256p % W;
      const bool ragged = rem != 0 && rem * 2 > W;
      const long long cost256 = (t256p + W - 1) / W * 256, cost224 = (t224p + W - 1) / W * 224;
      if (want_n == 224 || (want_n == 0 && ragged && cost224 * 100 < cost256 * 95)) tc_block_n = 224;
    }
    if (const char* env = std::getenv("GE_SPLIT_TAIL"))
      if (env[0] == '0') tc_split = false;
    if (backward) tc_split = false;  // their bias-gradient partials are per tile
    if (epi_is_norm(epi)) tc_split = false;  // the norm statistics are taken per whole tile
    // Eight epilogue warps for the GELU derivative, the heaviest epilogue:
    // with four it lengthens the GEMM (11008x8192x4096 with DGELU_BGRAD:
    // 0.555 ms with eight, 0.654 with four). Every other epilogue measured
    // faster with four (NONE 0.452 vs 0.478 ms on the same shape; the norm
    // fusion at 4096x8192x4096: 0.235 vs 0.241 ms).
    tmp.epi_warps = epi == GE_EPI_DGELU_BGRAD ? 8 : 4;
    // A problem of at most two waves has the epilogue of a CTA's last (or
    // only) tile on its critical path, overlapped with no MMA: eight warps
    // take it in about two thirds of the time (4096x2048x4096 GELU_BIAS:
    // 53.5 vs 55.1 us). With more waves four are faster (11008x8192x4096:
    // 425 vs 441 us).
    {
      const long long tm = tc_pair ? 256 : 128;
      const long long tiles = ((Mk + tm - 1) / tm) * ((Nk + tc_block_n - 1) / tc_block_n);
      const long long workers = tc_pair ? tmp.num_sms / 2 : tmp.num_sms;
      if (tiles <= 2 * workers) tmp.epi_warps = 8;
    }
    if (const char* env = std::getenv("GE_TWO_PRODUCERS")) tmp.two_producers = env[0] == '1' ? 1 : 0;
    if (const char* env = std::getenv("GE_EPI_WARPS")) {  // sweeps
      if (env[0] == '4') tmp.epi_warps = 4;
      if (env[0] == '8') tmp.epi_warps = 8;
    }
    if (dw_mask) tmp.epi_warps = 4;  // the masking warps take the place of four more
  }
  size_t ws = 256;
  size_t chain_x_off = 0;
  if (tmp.path == GE_PATH_GEMV || tmp.chain_ok) {
    ws += static_cast<size_t>(kChainSyncWords) * 4;  // ge_execute_chain
    if (tmp.chain_ok) {  // a plan a chain can run on: its exchange words
      ws = (ws + 255) / 256 * 256;
      chain_x_off = ws;
      ws += chain_xbuf_words(M, N) * 4;
      if (const char* env = std::getenv("GE_CHAIN_PRODUCERS")) tmp.chain_producers = std::atoi(env);  // sweeps
      if (const char* env = std::getenv("GE_CHAIN_INFLIGHT")) tmp.chain_inflight = std::atoi(env);
    }
  }
  size_t sk_off = 0;
  if (tmp.path == GE_PATH_TC_GEMM) {
    // stream-K: epoch, finished-CTA count, one flag per (CTA, epilogue warp)
    sk_off = ws;
    ws += (2 + 8 * static_cast<size_t>(tmp.num_sms)) * 4;
  }
  size_t bg_off = 0;
  if (tmp.path == GE_PATH_TC_GEMM && backward) {
    const int64_t Mk = tmp.swap ? N : M;
    const int64_t Nk = tmp.swap ? M : N;
    if (tmp.swap) {  // bgrad indexes D' columns: partials per 32-row block
      tmp.bg_rows = (Mk + 31) / 32;
      tmp.bg_len = Nk;
    } else {         // bgrad indexes D' rows: partials per n-tile and epilogue half (capacity: 128-wide tiles)
      tmp.bg_rows = 2 * ((Nk + 127) / 128);
      tmp.bg_len = Mk;
    }
    ws = (ws + 255) / 256 * 256;
    bg_off = ws;
    ws += static_cast<size_t>(tmp.bg_rows) * static_cast<size_t>(tmp.bg_len) * 4;
  }
  if (tmp.path == GE_PATH_TC_GEMM && dw_mask) {
    // bias-gradient partials: one row per split-K piece (at most 16) over M
    ws = (ws + 255) / 256 * 256;
    bg_off = ws;
    ws += 16 * static_cast<size_t>(M) * 4;
  }
  size_t nstats_off = 0, rowstats_off = 0;
  if (tmp.path == GE_PATH_TC_GEMM && epi_is_norm(epi)) {
    // D is column-major here, so the kernel's rows are the N tokens and its
    // columns the M features; capacity for the narrowest (128-wide) tiles.
    ws = (ws + 255) / 256 * 256;
    nstats_off = ws;
    ws += 2 * static_cast<size_t>((M + 127) / 128) * static_cast<size_t>(N) * 8;
    ws = (ws + 255) / 256 * 256;
    rowstats_off = ws;
    ws += static_cast<size_t>(N) * 8;
  }
  if (tmp.path == GE_PATH_DRELU && L.d == GE_D_COL) {
    tmp.splits = drelu_splits(tmp.R, tmp.C, tmp.num_sms, epi == GE_EPI_DGELU_BGRAD ? 1 : 0);
    const int64_t strips = (tmp.C + 255) / 256;
    ws += static_cast<size_t>(strips) * 4;
    ws = (ws + 255) / 256 * 256;
    ws += static_cast<size_t>(tmp.splits) * static_cast<size_t>(tmp.C) * 4;
  }
  if (cudaMalloc(&tmp.ws, ws) != cudaSuccess) {
    cudaGetLastError();
    return GE_ERR_OOM;
  }
  if (cudaMemset(tmp.ws, 0, ws) != cudaSuccess) {
    cudaFree(tmp.ws);
    cudaGetLastError();
    return GE_ERR_CUDA;
  }
  tmp.ws_bytes = ws;
  tmp.err = static_cast<unsigned int*>(tmp.ws);
  if (bg_off) tmp.bg_partials = reinterpret_cast<float*>(static_cast<char*>(tmp.ws) + bg_off);
  if (sk_off) tmp.sk_sync = reinterpret_cast<unsigned int*>(static_cast<char*>(tmp.ws) + sk_off);
  if (chain_x_off) tmp.chain_x = reinterpret_cast<unsigned int*>(static_cast<char*>(tmp.ws) + chain_x_off);
  if (nstats_off) {
    tmp.nstats = reinterpret_cast<float2*>(static_cast<char*>(tmp.ws) + nstats_off);
    tmp.rowstats = reinterpret_cast<float2*>(static_cast<char*>(tmp.ws) + rowstats_off);
  }
  if (tmp.path == GE_PATH_DRELU && L.d == GE_D_COL) {
    tmp.counters = reinterpret_cast<unsigned int*>(static_cast<char*>(tmp.ws) + 256);
    const int64_t strips = (tmp.C + 255) / 256;
    size_t off = 256 + static_cast<size_t>(strips) * 4;
    off = (off + 255) / 256 * 256;
    tmp.partials = reinterpret_cast<float*>(static_cast<char*>(tmp.ws) + off);
  }
  Plan* pl = new (std::nothrow) Plan(tmp);
  if (!pl) {
    cudaFree(tmp.ws);
    return GE_ERR_OOM;
  }
  if (pl->path == GE_PATH_TC_GEMM) {
    pl->tc_allow_split = tc_split;
    bool split_on = tc_split;
    bool tuned_kb64 = false;
    const bool overridden = std::getenv("GE_TILE_N") || std::getenv("GE_PAIR") || std::getenv("GE_SPLIT_TAIL") ||
                            std::getenv("GE_STREAM_K");
    if (!overridden) {
      std::lock_guard<std::mutex> lock(tuned_mutex());
      auto it = tuned_cache().find(tune_key(*pl));
      if (it != tuned_cache().end()) {
        tc_block_n = it->second.block_n;
        tc_pair = it->second.pair;
        split_on = tc_split && (it->second.split > 1 || it->second.sk);
        tuned_kb64 = it->second.kb == 64;
      }
    }
    ge_status_t st = apply_config(pl, tc_config(*pl, tc_block_n, tc_pair, split_on, tuned_kb64));
    if (st != GE_OK) {
      cudaFree(pl->ws);
      delete pl;
      return st;
    }
  }
  // DW_DRELU_BGRAD as two launches unless GE_DW_MASK = gemm asks for the
  // mask applied inside the GEMM (measured at 11008 x 4096 x 8192: 0.46 ms
  // for the two launches, 1.74 ms in one: the masking warps' shared-memory
  // pass and their hand-off to the MMA cost more than the dZ round trip).
  const char* dw_env = std::getenv("GE_DW_MASK");
  if (pl->path == GE_PATH_TC_GEMM && dw_mask && !(dw_env && dw_env[0] == 'g')) {
    const ge_layout_t Ld{GE_K_MAJOR, GE_MN_MAJOR, GE_D_COL, 0, 0, L.lda, L.ld_aux};
    const ge_layout_t Lg{GE_MN_MAJOR, L.b, GE_D_ROW, L.lda, L.ldb, L.ldd, 0};
    ge_plan_t hd = nullptr, hg = nullptr;
    ge_status_t st = ge_plan_create(&hd, M, K, 0, a, b, d, compute, GE_EPI_DRELU_BGRAD, &Ld);
    if (st == GE_OK) st = ge_plan_create(&hg, M, N, K, a, b, d, compute, GE_EPI_NONE, &Lg);
    const size_t dz_bytes = static_cast<size_t>(K) * static_cast<size_t>(L.lda) * 2;
    const size_t bg_off = (dz_bytes + 255) / 256 * 256;
    void* dz = nullptr;
    if (st == GE_OK && cudaMalloc(&dz, bg_off + static_cast<size_t>(M) * 4) != cudaSuccess) {
      cudaGetLastError();
      st = GE_ERR_OOM;
    }
    if (st != GE_OK) {
      ge_plan_free(hd);
      ge_plan_free(hg);
      ge_plan_free(reinterpret_cast<ge_plan_t>(pl));
      return st;
    }
    pl->sub_drelu = reinterpret_cast<Plan*>(hd);
    pl->sub_gemm = reinterpret_cast<Plan*>(hg);
    pl->dz_ws = dz;
    pl->bg_scratch = reinterpret_cast<float*>(static_cast<char*>(dz) + bg_off);
  }
  *out = reinterpret_cast<ge_plan_t>(pl);
  return GE_OK;
}

ge_status_t ge_execute(ge_plan_t plan, const void* A, const void* B, const void* bias, void* D,
                       void* aux, void* stream) {
  Plan* pl = reinterpret_cast<Plan*>(plan);
  if (!pl) return GE_ERR_INVALID_ARG;
  if (pl->sub_gemm) {
    // DW_DRELU_BGRAD as two launches: dZ = dY * mask (+ bgrad), then dW = dZ^T . B
    if (!A || !B || !D || !aux) return GE_ERR_INVALID_ARG;
    void* bg = bias ? const_cast<void*>(bias) : static_cast<void*>(pl->bg_scratch);
    ge_status_t s1 = ge_execute(reinterpret_cast<ge_plan_t>(pl->sub_drelu), A, nullptr, bg, pl->dz_ws, aux, stream);
    if (s1 != GE_OK) return s1;
    return ge_execute(reinterpret_cast<ge_plan_t>(pl->sub_gemm), pl->dz_ws, B, nullptr, D, nullptr, stream);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ge_status_t s;
  if (epi_is_norm(pl->epi)) return GE_ERR_UNSUPPORTED;  // ge_execute_norm
  if (pl->path == GE_PATH_DRELU) {
    // A = dY, D = dZ, aux = mask, bias = fp32 bgrad output.
    if (!A || !D || !aux || !bias) return GE_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(D) || !aligned16(aux) || !aligned16(bias)) return GE_ERR_ALIGNMENT;
    if ((s = check_device(pl, 0, A)) != GE_OK || (s = check_device(pl, 3, D)) != GE_OK ||
        (s = check_device(pl, 4, aux)) != GE_OK || (s = check_device(pl, 2, bias)) != GE_OK)
      return s;
    DreluArgs d{};
    d.R = pl->R;
    d.C = pl->C;
    d.dY = static_cast<const __half*>(A);
    d.dZ = static_cast<__half*>(D);
    d.ld = pl->L.ldd;
    d.mask = static_cast<const uint32_t*>(aux);
    d.ld_aux = pl->aux_words;
    d.bgrad = static_cast<float*>(const_cast<void*>(bias));
    d.partials = pl->partials;
    d.counters = pl->counters;
    d.splits = pl->splits;
    d.bf16 = pl->bf16;
    if (pl->epi == GE_EPI_DGELU_BGRAD) {  // aux is the stored pre-activation z
      d.gelu = 1;
      d.mask = nullptr;
      d.zaux = static_cast<const unsigned short*>(aux);
      d.ld_zaux = pl->aux_words;
    }
    cudaError_t e = launch_drelu_bgrad(d, pl->L.d == GE_D_COL ? 1 : 0, st);
    return e == cudaSuccess ? GE_OK : GE_ERR_CUDA;
  }
  if (!A || !B || !D) return GE_ERR_INVALID_ARG;
  if (pl->epi == GE_EPI_DRELU_BGRAD || pl->epi == GE_EPI_DGELU_BGRAD) {
    // GEMM-epilogue form: aux = forward mask or z (input), bias = fp32 bgrad output.
    if (!aux || !bias) return GE_ERR_INVALID_ARG;
    const uintptr_t aux_align = pl->epi == GE_EPI_DGELU_BGRAD ? 15u : 3u;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) || !aligned16(bias) ||
        (reinterpret_cast<uintptr_t>(aux) & aux_align))
      return GE_ERR_ALIGNMENT;
    if ((s = check_device(pl, 0, A)) != GE_OK || (s = check_device(pl, 1, B)) != GE_OK ||
        (s = check_device(pl, 3, D)) != GE_OK || (s = check_device(pl, 2, bias)) != GE_OK ||
        (s = check_device(pl, 4, aux)) != GE_OK)
      return s;
    return launch_forward(pl, A, B, bias, D, aux, static_cast<int>(pl->epi), st);
  }
  if (pl->epi == GE_EPI_DW_DRELU_BGRAD) {
    // A = dY, aux = the forward mask (input), bias = fp32 bgrad output or NULL.
    if (!aux) return GE_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) || !aligned16(aux) || (bias && !aligned16(bias)))
      return GE_ERR_ALIGNMENT;
    if ((s = check_device(pl, 0, A)) != GE_OK || (s = check_device(pl, 1, B)) != GE_OK ||
        (s = check_device(pl, 3, D)) != GE_OK || (s = check_device(pl, 4, aux)) != GE_OK ||
        (bias && (s = check_device(pl, 2, bias)) != GE_OK))
      return s;
    return launch_forward(pl, A, B, bias, D, aux, EPI_NONE, st);
  }
  if (epi_has_bias(pl->epi) && !bias) return GE_ERR_INVALID_ARG;
  const bool needs_aux = pl->epi == GE_EPI_RELU_AUX_BIAS || pl->epi == GE_EPI_GELU_AUX_BIAS;
  if (needs_aux && !aux) return GE_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B)) return GE_ERR_ALIGNMENT;
  if (pl->epi == GE_EPI_GELU_AUX_BIAS && !aligned16(aux)) return GE_ERR_ALIGNMENT;
  if (pl->path == GE_PATH_TC_GEMM && !aligned16(D)) return GE_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(D) & 1u) || (bias && (reinterpret_cast<uintptr_t>(bias) & 1u)) ||
      (aux && (reinterpret_cast<uintptr_t>(aux) & 3u)))
    return GE_ERR_ALIGNMENT;
  if ((s = check_device(pl, 0, A)) != GE_OK || (s = check_device(pl, 1, B)) != GE_OK ||
      (s = check_device(pl, 3, D)) != GE_OK)
    return s;
  if (epi_has_bias(pl->epi) && (s = check_device(pl, 2, bias)) != GE_OK) return s;
  if (needs_aux && (s = check_device(pl, 4, aux)) != GE_OK) return s;
  return launch_forward(pl, A, B, epi_has_bias(pl->epi) ? bias : nullptr, D, needs_aux ? aux : nullptr,
                        static_cast<int>(pl->epi), st);
}

ge_status_t ge_execute_unfused(ge_plan_t plan, const void* A, const void* B, const void* bias,
                               void* D, void* aux, void* stream) {
  Plan* pl = reinterpret_cast<Plan*>(plan);
  if (!pl) return GE_ERR_INVALID_ARG;
  if (!epi_has_bias(pl->epi) || pl->path == GE_PATH_DRELU || epi_is_norm(pl->epi)) return GE_ERR_UNSUPPORTED;
  if (!A || !B || !D || !bias) return GE_ERR_INVALID_ARG;
  const bool needs_aux = pl->epi == GE_EPI_RELU_AUX_BIAS || pl->epi == GE_EPI_GELU_AUX_BIAS;
  if (needs_aux && !aux) return GE_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(D)) return GE_ERR_ALIGNMENT;
  if (pl->L.ldd % 8 != 0) return GE_ERR_ALIGNMENT;
  if (pl->epi == GE_EPI_GELU_AUX_BIAS && !aligned16(aux)) return GE_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(bias) & 1u) || (aux && (reinterpret_cast<uintptr_t>(aux) & 3u)))
    return GE_ERR_ALIGNMENT;
  ge_status_t s;
  if ((s = check_device(pl, 0, A)) != GE_OK || (s = check_device(pl, 1, B)) != GE_OK ||
      (s = check_device(pl, 3, D)) != GE_OK || (s = check_device(pl, 2, bias)) != GE_OK)
    return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  s = launch_forward(pl, A, B, nullptr, D, nullptr, EPI_NONE, st);
  if (s != GE_OK) return s;
  __half* Dh = static_cast<__half*>(D);
  cudaError_t e = launch_bias_add(Dh, pl->R, pl->C, pl->L.ldd, static_cast<const __half*>(bias),
                                  pl->L.d == GE_D_ROW ? 1 : 0, pl->bf16, st);
  if (e != cudaSuccess) return GE_ERR_CUDA;
  if (pl->epi != GE_EPI_BIAS) {
    const bool zout = pl->epi == GE_EPI_GELU_AUX_BIAS;
    e = launch_activation(Dh, pl->R, pl->C, pl->L.ldd, static_cast<int>(pl->epi),
                          pl->epi == GE_EPI_RELU_AUX_BIAS ? static_cast<uint32_t*>(aux) : nullptr,
                          pl->aux_words, zout ? static_cast<unsigned short*>(aux) : nullptr,
                          pl->aux_words, pl->bf16, st);
    if (e != cudaSuccess) return GE_ERR_CUDA;
  }
  return GE_OK;
}

ge_status_t ge_execute_norm(ge_plan_t plan, const void* A, const void* B, const void* bias,
                            const void* residual, const void* gamma, const void* beta, void* H, void* Y,
                            float eps, void* stream) {
  Plan* pl = reinterpret_cast<Plan*>(plan);
  ge_status_t s = check_norm_args(pl, A, B, bias, residual, gamma, beta, H, Y);
  if (s != GE_OK) return s;
  if (!(eps >= 0.0f)) return GE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // h = A.B + bias + residual in the GEMM (or GEMV) epilogue, stored once as H
  s = launch_forward(pl, A, B, bias, H, const_cast<void*>(residual), EPI_BIAS_RESIDUAL, st);
  if (s != GE_OK) return s;
  return launch_norm_pass(pl, gamma, beta, H, Y, eps, pl->path == GE_PATH_TC_GEMM, st);
}

ge_status_t ge_execute_norm_unfused(ge_plan_t plan, const void* A, const void* B, const void* bias,
                                    const void* residual, const void* gamma, const void* beta, void* H,
                                    void* Y, float eps, void* stream) {
  Plan* pl = reinterpret_cast<Plan*>(plan);
  ge_status_t s = check_norm_args(pl, A, B, bias, residual, gamma, beta, H, Y);
  if (s != GE_OK) return s;
  if (!(eps >= 0.0f)) return GE_ERR_INVALID_ARG;
  if (H == residual) return GE_ERR_INVALID_ARG;  // the GEMM writes H before the residual is added
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  s = launch_forward(pl, A, B, nullptr, H, nullptr, EPI_NONE, st);
  if (s != GE_OK) return s;
  __half* Hh = static_cast<__half*>(H);
  if (launch_bias_add(Hh, pl->R, pl->C, pl->L.ldd, static_cast<const __half*>(bias), 0, pl->bf16, st) !=
      cudaSuccess)
    return GE_ERR_CUDA;
  if (launch_residual_add(Hh, pl->R, pl->C, pl->L.ldd, static_cast<const unsigned short*>(residual), pl->bf16,
                          st) != cudaSuccess)
    return GE_ERR_CUDA;
  return launch_norm_pass(pl, gamma, beta, H, Y, eps, false, st);
}

ge_status_t ge_execute_chain(ge_plan_t plan, int64_t layers, const void* const* A, const void* const* bias,
                             const void* X, void* Y, void* stream) {
  Plan* pl = reinterpret_cast<Plan*>(plan);
  if (!pl) return GE_ERR_INVALID_ARG;
  // a decode-sized plan whose layers can feed one another: square, the
  // output stored like the next layer's input (D column-major: N rows of M)
  if (!pl->chain_ok) return GE_ERR_UNSUPPORTED;
  if (pl->K % 8 != 0 || pl->L.ldd % 8 != 0 || pl->L.ldb % 8 != 0) return GE_ERR_ALIGNMENT;
  // the activations and one weight-row segment must fit in shared memory
  if (gemv_chain_slots(static_cast<int>(pl->K), static_cast<int>(pl->N)) < 1) return GE_ERR_UNSUPPORTED;
  if (layers < 1 || layers > kChainMaxLayers) return GE_ERR_INVALID_ARG;
  const bool has_bias = pl->epi != GE_EPI_NONE;
  if (!A || !X || !Y || (has_bias && !bias)) return GE_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Y)) return GE_ERR_ALIGNMENT;
  for (int64_t l = 0; l < layers; ++l) {
    if (!A[l] || (has_bias && !bias[l])) return GE_ERR_INVALID_ARG;
    if (!aligned16(A[l]) || (has_bias && (reinterpret_cast<uintptr_t>(bias[l]) & 1u))) return GE_ERR_ALIGNMENT;
  }
  ge_status_t s;
  if ((s = check_device(pl, 1, X)) != GE_OK || (s = check_device(pl, 3, Y)) != GE_OK) return s;
  for (int64_t l = 0; l < 2 * layers; ++l) {
    const void* p = l < layers ? A[l] : (has_bias ? bias[l - layers] : nullptr);
    if (!p) continue;
    const unsigned long long id = buffer_id(p);
    auto it = pl->chain_checked.find(p);
    if (it != pl->chain_checked.end() && id != 0 && it->second == id) continue;
    if ((s = check_device(pl, 5, p)) != GE_OK) return s;
    if (pl->chain_checked.size() > 4096) pl->chain_checked.clear();
    pl->chain_checked[p] = id;
  }
  ChainArgs c{};
  c.layers = static_cast<int>(layers);
  c.M = static_cast<int>(pl->M);
  c.K = static_cast<int>(pl->K);
  c.N = static_cast<int>(pl->N);
  for (int64_t l = 0; l < layers; ++l) {
    c.A[l] = static_cast<const unsigned short*>(A[l]);
    c.bias[l] = has_bias ? static_cast<const unsigned short*>(bias[l]) : nullptr;
  }
  c.lda = pl->L.lda;
  c.X = static_cast<const unsigned short*>(X);
  c.ldx = pl->L.ldb;
  c.Y = static_cast<unsigned short*>(Y);
  c.ldy = pl->L.ldd;
  c.epi = static_cast<int>(pl->epi);
  c.bf16 = pl->bf16;
  c.err = pl->err;
  c.sync = reinterpret_cast<unsigned int*>(static_cast<char*>(pl->ws) + 256);
  c.xbuf = pl->chain_x;
  c.producers = pl->chain_producers;
  c.inflight = pl->chain_inflight;
  if (!c.xbuf) return GE_ERR_UNSUPPORTED;
  c.budget = kWaitBudgetCycles;
  const cudaError_t e = launch_gemv_chain(c, pl->num_sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GE_OK : GE_ERR_CUDA;
}

void ge_autotune_cache_clear(void) {
  std::lock_guard<std::mutex> lock(tuned_mutex());
  tuned_cache().clear();
}

ge_status_t ge_plan_autotune(ge_plan_t plan, const void* A, const void* B, const void* bias, void* D,
                             void* aux, void* stream, int reps) {
  Plan* pl = reinterpret_cast<Plan*>(plan);
  if (!pl || reps < 1 || reps > 1000) return GE_ERR_INVALID_ARG;
  if (pl->path != GE_PATH_TC_GEMM) return GE_OK;  // nothing to choose
  if (pl->sub_gemm) {  // two launches: tune the GEMM on this call's dZ
    if (!A || !B || !D || !aux) return GE_ERR_INVALID_ARG;
    void* bg = bias ? const_cast<void*>(bias) : static_cast<void*>(pl->bg_scratch);
    ge_status_t s1 = ge_execute(reinterpret_cast<ge_plan_t>(pl->sub_drelu), A, nullptr, bg, pl->dz_ws, aux, stream);
    if (s1 != GE_OK) return s1;
    return ge_plan_autotune(reinterpret_cast<ge_plan_t>(pl->sub_gemm), pl->dz_ws, B, nullptr, D, nullptr, stream,
                            reps);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const TcConfig current = tc_config(*pl, pl->block_n, pl->pair, pl->split > 1 || pl->tc_allow_split, pl->kb == 64);
  // tile width x pair mode x split tail (or stream-K) on / off x stage
  // shape (two 64-wide k panels a stage where they fit, or one)
  TcConfig cands[16];
  int n = 0;
  const bool b_mn_k = pl->swap ? (pl->L.a == GE_MN_MAJOR) : (pl->L.b == GE_MN_MAJOR);
  for (int bn : {128, 256, 224})
    for (int pair : {0, 1}) {
      if (pair && bn == 128) continue;
      if (bn == 224 && (!pair || b_mn_k || pl->epi == GE_EPI_DW_DRELU_BGRAD)) continue;
      for (bool kb64 : {false, true}) {
        const TcConfig c0 = tc_config(*pl, bn, pair, false, kb64);
        if (kb64 && c0.kb == tc_config(*pl, bn, pair, false).kb) continue;  // one panel already
        cands[n++] = c0;
        if (pl->tc_allow_split) {
          const TcConfig c = tc_config(*pl, bn, pair, true, kb64);
          if (c.split > 1 || c.sk_tiles > 0) cands[n++] = c;
        }
      }
    }
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    cudaGetLastError();
    return GE_ERR_CUDA;
  }
  int best = -1;
  float best_ms = 0.0f;
  ge_status_t s = GE_OK;
  for (int i = 0; i < n && s == GE_OK; ++i) {
    if ((s = apply_config(pl, cands[i])) != GE_OK) break;
    if ((s = ge_execute(plan, A, B, bias, D, aux, stream)) != GE_OK) break;  // warm-up, checks args
    cudaEventRecord(e0, st);
    for (int r = 0; r < reps && s == GE_OK; ++r) s = ge_execute(plan, A, B, bias, D, aux, stream);
    cudaEventRecord(e1, st);
    if (cudaEventSynchronize(e1) != cudaSuccess) {
      cudaGetLastError();
      s = GE_ERR_CUDA;
      break;
    }
    float ms = 0.0f;
    cudaEventElapsedTime(&ms, e0, e1);
    if (best < 0 || ms < best_ms) {
      best = i;
      best_ms = ms;
    }
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  const ge_status_t s2 = apply_config(pl, best >= 0 ? cands[best] : current);
  if (s != GE_OK) return s;
  if (s2 != GE_OK) return s2;
  {
    std::lock_guard<std::mutex> lock(tuned_mutex());
    tuned_cache()[tune_key(*pl)] =
        TunedChoice{cands[best].block_n, cands[best].pair, cands[best].split, cands[best].sk_tiles > 0 ? 1 : 0,
                    cands[best].kb};
  }
  return ge_execute(plan, A, B, bias, D, aux, stream);  // outputs of the chosen configuration
}

int ge_plan_config(ge_plan_t plan, int* block_n, int* pair, int* split) {
  Plan* pl = reinterpret_cast<Plan*>(plan);
  if (!pl) return -1;
  if (pl->sub_gemm) return ge_plan_config(reinterpret_cast<ge_plan_t>(pl->sub_gemm), block_n, pair, split);
  if (block_n) *block_n = pl->path == GE_PATH_TC_GEMM ? pl->block_n : 0;
  if (pair) *pair = pl->path == GE_PATH_TC_GEMM ? pl->pair : 0;
  if (split) *split = pl->path == GE_PATH_TC_GEMM ? pl->split : 0;
  return static_cast<int>(pl->path);
}

int ge_plan_stream_k_tiles(ge_plan_t plan) {
  Plan* pl = reinterpret_cast<Plan*>(plan);
  if (!pl) return -1;
  if (pl->sub_gemm) return ge_plan_stream_k_tiles(reinterpret_cast<ge_plan_t>(pl->sub_gemm));
  return pl->path == GE_PATH_TC_GEMM ? pl->sk_tiles : 0;
}

ge_status_t ge_plan_set_attr(ge_plan_t plan, ge_plan_attr_t attr, int64_t value) {
  Plan* pl = reinterpret_cast<Plan*>(plan);
  if (!pl) return GE_ERR_INVALID_ARG;
  switch (attr) {
    case GE_ATTR_STATIC_A:
      if (value != 0 && value != 1) return GE_ERR_INVALID_ARG;
      pl->static_a = static_cast<int>(value);
      return GE_OK;
  }
  return GE_ERR_INVALID_ARG;
}

ge_status_t ge_plan_free(ge_plan_t plan) {
  Plan* pl = reinterpret_cast<Plan*>(plan);
  if (!pl) return GE_OK;
  ge_status_t s = GE_OK;
  if (pl->ws && cudaFree(pl->ws) != cudaSuccess) {
    cudaGetLastError();
    s = GE_ERR_CUDA;
  }
  if (pl->tail_ws && cudaFree(pl->tail_ws) != cudaSuccess) {
    cudaGetLastError();
    s = GE_ERR_CUDA;
  }
  if (pl->dz_ws && cudaFree(pl->dz_ws) != cudaSuccess) {
    cudaGetLastError();
    s = GE_ERR_CUDA;
  }
  const ge_status_t s1 = ge_plan_free(reinterpret_cast<ge_plan_t>(pl->sub_drelu));
  const ge_status_t s2 = ge_plan_free(reinterpret_cast<ge_plan_t>(pl->sub_gemm));
  delete pl;
  return s != GE_OK ? s : (s1 != GE_OK ? s1 : s2);
}

size_t ge_aux_bytes(ge_plan_t plan) {
  Plan* pl = reinterpret_cast<Plan*>(plan);
  if (!pl) return 0;
  if (pl->epi == GE_EPI_RELU_AUX_BIAS)
    return static_cast<size_t>(pl->R) * static_cast<size_t>(pl->aux_words) * 4u;
  if (pl->epi == GE_EPI_GELU_AUX_BIAS)
    return static_cast<size_t>(pl->R) * static_cast<size_t>(pl->aux_words) * 2u;
  return 0;
}

int64_t ge_aux_ld(ge_plan_t plan) {
  Plan* pl = reinterpret_cast<Plan*>(plan);
  return pl ? pl->aux_words : 0;
}

int ge_plan_path(ge_plan_t plan) {
  Plan* pl = reinterpret_cast<Plan*>(plan);
  return pl ? static_cast<int>(pl->path) : -1;
}

int ge_plan_tile_n(ge_plan_t plan) {
  Plan* pl = reinterpret_cast<Plan*>(plan);
  if (pl && pl->sub_gemm) return ge_plan_tile_n(reinterpret_cast<ge_plan_t>(pl->sub_gemm));
  return (pl && pl->path == GE_PATH_TC_GEMM) ? pl->block_n : 0;
}

ge_status_t ge_get_last_device_error(ge_plan_t plan) {
  Plan* pl = reinterpret_cast<Plan*>(plan);
  if (!pl) return GE_ERR_INVALID_ARG;
  unsigned int w = 0;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(&w, pl->err, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(pl->err, 0, sizeof(w)) != cudaSuccess) {
    cudaGetLastError();
    return GE_ERR_CUDA;
  }
  ge_status_t s = (w & ERR_DEBUG_CHECK) ? GE_ERR_DEVICE_CHECK : (w ? GE_ERR_TIMEOUT : GE_OK);
  // a plan run as two launches: their own words too (the gravest status wins:
  // a failed read, then a failed check, then an expired wait)
  auto rank = [](ge_status_t x) { return x == GE_ERR_CUDA ? 3 : x == GE_ERR_DEVICE_CHECK ? 2 : x == GE_ERR_TIMEOUT ? 1 : 0; };
  for (Plan* sub : {pl->sub_drelu, pl->sub_gemm}) {
    if (!sub) continue;
    const ge_status_t t = ge_get_last_device_error(reinterpret_cast<ge_plan_t>(sub));
    if (rank(t) > rank(s)) s = t;
  }
  return s;
}

ge_status_t ge_debug_wait_timeout(ge_plan_t plan, int64_t budget_cycles, void* stream) {
  Plan* pl = reinterpret_cast<Plan*>(plan);
  if (!pl || budget_cycles < 1 || budget_cycles > (int64_t(1) << 31)) return GE_ERR_INVALID_ARG;
  cudaError_t e = launch_wait_probe(pl->err, budget_cycles, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GE_OK : GE_ERR_CUDA;
}

int ge_debug_checks(void) {
#ifdef GE_DEBUG
  return 1;
#else
  return 0;
#endif
}

ge_status_t ge_debug_check_probe(ge_plan_t plan, void* stream) {
  Plan* pl = reinterpret_cast<Plan*>(plan);
  if (!pl) return GE_ERR_INVALID_ARG;
  const cudaError_t e = launch_check_probe(pl->err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GE_OK : GE_ERR_CUDA;
}

}  // extern "C"
