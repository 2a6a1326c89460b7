// ge_internal.h -- declarations shared by the library's translation units
// (host planner <-> kernel launchers). Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace ge {

// Epilogue codes used by the kernels.
enum EpiCode : int {
  EPI_NONE = 0,
  EPI_BIAS = 1,
  EPI_RELU_BIAS = 2,
  EPI_GELU_BIAS = 3,
  EPI_RELU_AUX_BIAS = 4,
  EPI_DRELU_BGRAD = 5,  // GEMM epilogue form: aux is the input mask
  EPI_GELU_ERF_BIAS = 6,
  EPI_GELU_AUX_BIAS = 7,  // tanh-GELU; the pre-activation z is a second output (zaux)
  EPI_DGELU_BGRAD = 8,    // GEMM epilogue form: zaux is the input pre-activation
  EPI_BIAS_RESIDUAL = 9   // h = A.B + bias + residual (zaux is the residual input)
};

// Device error word bits (the plan's workspace word 0).
enum ErrBits : unsigned int {
  ERR_PRODUCER_TIMEOUT = 1u,
  ERR_MMA_TIMEOUT = 2u,
  ERR_EPILOGUE_TIMEOUT = 4u,
  ERR_DRAIN_TIMEOUT = 8u,
  ERR_PROBE_TIMEOUT = 16u,
  ERR_XFORM_TIMEOUT = 32u,
  ERR_CHAIN_TIMEOUT = 64u,
  ERR_DEBUG_CHECK = 128u,  // a GE_DEBUG build's index / offset / phase check failed
  ERR_PEER_TIMEOUT = 256u  // a stream-K tile's finisher waited too long for a peer's piece
};

// Checks of the GE_DEBUG build: a failed check records ERR_DEBUG_CHECK in
// the error word and evaluates to false, so the caller skips the access (a
// skipped copy then ends in a bounded wait that aborts the kernel). No trap,
// no assert: the context stays usable. Without GE_DEBUG it is `true`.
#ifdef GE_DEBUG
#define GE_DCHECK(cond, errp) ((cond) ? true : (atomicOr((errp), ::ge::ERR_DEBUG_CHECK), false))
#else
#define GE_DCHECK(cond, errp) true
#endif

// Kernel-level problem of the tensor-core GEMM: D'[Mk, Nk] (row-major, via
// the D tensor map) = act(A'[Mk, K] . B'[K, Nk] + bias), where the planner
// has already folded a column-major D into swapped operands.
struct GemmArgs {
  int Mk, Nk, K;
  int a_mn;          // A' is M-major (1) or K-major (0)
  int b_mn;          // B' is N-major (1) or K-major (0)
  int epi;           // EpiCode
  int bf16;          // element type of A, B, bias, D: bfloat16 (1) or fp16 (0)
  int bias_per_col;  // bias indexed by D' column (1) or row (0)
  const __half* bias;
  uint32_t* aux;     // mask words, rows of D', ld_aux words per row
  long long ld_aux;
  __half* D;         // D' base (row-major, ldd elements per row): ragged-edge stores
  long long ldd;
  unsigned int* err; // device error word
  int group_m;       // tile rasterisation group (m-tiles per group)
  int two_producers;  // 1: a second producer warp issues the B loads
  long long budget;  // bounded-wait budget in SM clock cycles
  // Split-K tail: tiles >= tail_start are computed as `split` k-ranges whose
  // fp32 accumulators go to `partials` ([tile - tail_start][split][TILE_M][BN]);
  // tc_gemm_fixup then adds them in split order and applies the epilogue.
  int tail_start;
  int split;
  float* partials;
  // D*_BGRAD epilogue: per-block bias-gradient partial sums, reduced by
  // launch_bgrad_reduce into `bgrad`. Row case (bias per D' row): bg_partials
  // is [halves * num n-tiles][Mk] (per n-tile, one row for each epilogue
  // warp of a lane quarter: halves = epi_warps / 4); column case:
  // [ceil(Mk/32)][Nk].
  float* bg_partials;
  float* bgrad;
  // GELU_AUX_BIAS: z of every element, written like D' (ld_zaux elements per
  // row; through the zaux tensor map except on a ragged edge). DGELU_BGRAD:
  // the stored z read back (same layout). BIAS_RESIDUAL: the residual input
  // (same layout; it may be D itself).
  unsigned short* zaux;
  long long ld_zaux;
  // BIAS_RESIDUAL: statistics of h per (n-tile, D' row) over the columns of
  // the tile's 32-column slabs c with c % halves == half: (mean, sum of
  // squared deviations) as float2 at nstats[(halves * nt + half) * Mk + row];
  // null = not wanted.
  float2* nstats;
  // DW_DRELU_BGRAD (amask = 1): A' (M-major) is masked by the forward's ReLU
  // mask as it is loaded (the mask arrives through the fourth tensor map);
  // with bg_partials set, the masked A' is also summed over each unit's
  // k-range into bg_partials[piece][Mk] (piece = split-K piece, 0 for whole
  // tiles, whose other rows are zeroed), by the CTAs of the first N-tile.
  int amask;
  // k-values per pipeline stage: 64, or 128 (two 64-wide panels per operand
  // box; K-major operands then come through 3-D tensor maps that index the
  // panels, so K must be a multiple of 128)
  int kb;
  // Stream-K (sk_tiles > 0; then split = 1 and there is no split-K tail):
  // the last sk_tiles tiles are cut into I = sk_tiles * ceil(K / kb)
  // k-block iterations, and worker w of the W = grid / (pair ? 2 : 1)
  // workers computes iterations [w * I / W, (w + 1) * I / W) after its
  // share of the other tiles. A worker's first stream-K segment, when it
  // starts inside a tile, goes as fp32 to slot w of `partials`
  // ([W][TILE_M][BN]); the worker whose segment starts the tile adds the
  // slots of the tile's other segments in k order in its epilogue.
  // sk_sync: [0] launch epoch, [1] finished-CTA count, [2 + cta * epi_warps
  // + warp] the epoch + 1 at which that epilogue warp's rows of the CTA's
  // slot are complete. Zeroed once; every launch leaves it consistent.
  int sk_tiles;
  unsigned int* sk_sync;
};

// pair = 1: 2-CTA clusters (cta_group::2, 256-row tiles); grid counts CTAs
// (even) and the B tensor map's box is BN/2 rows (K-major B). epi_warps = 4
// or 8 epilogue warps (8: two per TMEM lane quarter on alternate slabs; the
// D*_BGRAD row partials and the norm statistics then have two halves per
// n-tile).
int tc_gemm_max_pairs(int block_n, int num_sms, int epi_warps);
cudaError_t launch_tc_gemm_fixup(int block_n, int pair, const GemmArgs& args, int num_sms, cudaStream_t stream);
// out[i] = sum over j = 0..rows-1 of part[j * len + i] in fp32, in a fixed
// order: for each w = 0..7 the rows j = w, w + 8, w + 16, ... are added in
// turn, then the eight sums are added in w order (the same result every run).
cudaError_t launch_bgrad_reduce(const float* part, long long rows, long long len, float* out,
                                cudaStream_t stream);
// tmZ: the zaux tensor map (GELU_AUX_BIAS; any valid map otherwise).
cudaError_t launch_tc_gemm(int block_n, int pair, int epi_warps, const CUtensorMap& tmA,
                           const CUtensorMap& tmB, const CUtensorMap& tmD, const CUtensorMap& tmZ,
                           const GemmArgs& args, int grid, cudaStream_t stream);

// Weight-streaming GEMV for N <= 16: A K-major [M, K] (lda), B K-major
// (B[k,n] at B[n*ldb + k]), D[m,n] at m*ldd_m + n*ldd_n.
struct GemvArgs {
  int M, N, K;
  const __half* A;
  long long lda;
  const __half* B;
  long long ldb;
  __half* D;
  long long ldd_m, ldd_n;
  const __half* bias;
  const unsigned short* res;  // BIAS_RESIDUAL: residual, strides as D (may be D)
  int epi;
  int bf16;           // element type: bfloat16 (1) or fp16 (0)
  int static_a;       // launch with programmatic dependent launch (A never written upstream)
  unsigned int* err;  // device error word (GE_DEBUG checks)
};
cudaError_t launch_gemv(const GemvArgs& args, int num_sms, cudaStream_t stream);

// A stack of `layers` square decode projections in one cooperative launch:
// Y_0 = act(A_0 . X + bias_0), Y_l = act(A_l . Y_(l-1) + bias_l), each Y_l
// rounded to the element type. X is [N][ldx], layer l's output is
// Y + l * N * ldy, [N][ldy] (N tokens of M = K features).
constexpr int kChainMaxLayers = 64;
// Synchronisation words of a chain in the plan workspace: the launch epoch
// (advanced by the last block of every launch), the finished-block count,
// the abort flag and one arrival count per layer (all but the epoch zero
// between launches).
constexpr int kChainSyncWords = 3 + kChainMaxLayers;
// Exchange words of a chain (2 x N x M, in the workspace of plans a chain
// can run on): each layer's outputs, 16-bit value in the low half and a
// (launch, layer) tag in the high half, double-buffered by layer parity.
inline size_t chain_xbuf_words(long long M, long long N) { return 2ull * static_cast<size_t>(M * N); }
struct ChainArgs {
  int layers, M, K, N;
  const unsigned short* A[kChainMaxLayers];     // [M][lda] each
  const unsigned short* bias[kChainMaxLayers];  // [M] each; unused for EPI_NONE
  long long lda;
  const unsigned short* X;
  long long ldx;
  unsigned short* Y;
  long long ldy;
  int epi;
  int bf16;
  int slots;                // (set by the launcher) weight-segment slots per block
  int producers;            // producer warps per block (0: the launcher's choice)
  int inflight;             // bulk copies in flight per block (0: the launcher's choice)
  unsigned int* err;        // device error word
  unsigned int* sync;       // kChainSyncWords words
  unsigned int* xbuf;       // 2 x N x M tagged activation words (the layers' exchange)
  long long budget;         // bounded-wait budget in SM clock cycles
};
// Weight-segment slots per block that fit in shared memory beside the
// staged activations (0: not even one).
int gemv_chain_slots(int K, int N);
cudaError_t launch_gemv_chain(const ChainArgs& args, int num_sms, cudaStream_t stream);

// DRELU_BGRAD (gelu = 0: mask bits) or DGELU_BGRAD (gelu = 1: the stored
// pre-activation zaux) on a stored matrix of R rows x C contiguous columns.
// reduce_rows = 1: bgrad[c] = sum over rows r (D column-major case);
// reduce_rows = 0: bgrad[r] = sum over columns c (D row-major case).
struct DreluArgs {
  long long R, C;
  const __half* dY;
  __half* dZ;
  long long ld;       // elements
  const uint32_t* mask;
  long long ld_aux;   // words
  float* bgrad;
  float* partials;    // [splits][C] workspace (reduce_rows only)
  unsigned int* counters;  // [ceil(C/256)] workspace (reduce_rows only)
  int splits;
  int bf16;           // element type of dY / dZ: bfloat16 (1) or fp16 (0)
  int gelu;           // DGELU_BGRAD: dZ = dY * gelu'(z) with z from zaux
  const unsigned short* zaux;
  long long ld_zaux;  // elements
};
cudaError_t launch_drelu_bgrad(const DreluArgs& args, int reduce_rows, cudaStream_t stream);
int drelu_splits(long long R, long long C, int num_sms, int gelu);

// Unfused baseline kernels, in place on D (R rows x C contiguous, ld).
cudaError_t launch_bias_add(__half* D, long long R, long long C, long long ld, const __half* bias,
                            int bias_per_row, int bf16, cudaStream_t stream);
// GELU_AUX_BIAS also copies z to zaux (ld_zaux elements per row) first.
cudaError_t launch_activation(__half* D, long long R, long long C, long long ld, int epi,
                              uint32_t* aux, long long ld_aux, unsigned short* zaux,
                              long long ld_zaux, int bf16, cudaStream_t stream);

// Normalisation of every row of H (R rows x C contiguous features, ld):
// RMSNorm (layer = 0) y = h * rsqrt(mean(h^2) + eps) * gamma, or LayerNorm
// (layer = 1) y = (h - mean) * rsqrt(var + eps) * gamma + beta (population
// variance), written to Y (same layout; Y may be H).
struct NormArgs {
  long long R, C, ld;
  const unsigned short* H;
  unsigned short* Y;
  const unsigned short* gamma;
  const unsigned short* beta;
  float eps;
  int layer;
  int bf16;
  // Statistics already taken by the GEMM epilogue (GemmArgs::nstats):
  // partials [halves * ntiles][R] for tiles tile_w features wide (the
  // 32-feature slabs c % halves == half of each tile); rowstats ([R],
  // scratch) receives (mean, rstd). partials == null: the pass takes them
  // itself.
  const float2* partials;
  int ntiles, tile_w, halves;
  float2* rowstats;
};
cudaError_t launch_norm(const NormArgs& args, int num_sms, cudaStream_t stream);
// D[r, c] += res[r * ld + c] (unfused baseline of the residual add).
cudaError_t launch_residual_add(__half* D, long long R, long long C, long long ld,
                                const unsigned short* res, int bf16, cudaStream_t stream);

// Bounded-wait probe (test hook).
cudaError_t launch_wait_probe(unsigned int* err, long long budget, cudaStream_t stream);
// Debug-check probe (test hook): records ERR_DEBUG_CHECK in a GE_DEBUG build.
cudaError_t launch_check_probe(unsigned int* err, cudaStream_t stream);

}  // namespace ge
