/*
 * ge.h -- C ABI of the GB300 fused linear-layer engine (libgemm_epilogues.so).
 *
 * One operation family: D = act(A.B + bias) computed as a single GEMM whose
 * epilogue adds a broadcast bias vector and applies an activation in
 * registers before one store of D, plus the matching backward epilogue.
 *
 * Sources (page title, section) for what each call computes:
 *  - nvmath-python cuBLASLt bias-fusion guide, "Core API and parameter
 *    configuration": the plan -> execute -> free life cycle; weights (m,k)
 *    times x (k,n) plus a bias of shape (m,1) broadcast over the n columns;
 *    fp16 operands with a 32-bit compute type and fp16 output.
 *  - same page, "Advanced techniques": RELU_BIAS and GELU_BIAS fuse the
 *    activation after the bias; DRELU_BGRAD fuses the ReLU-gradient mask with
 *    the bias-gradient accumulation in the backward pass (also the source of
 *    DW_DRELU_BGRAD, which applies that mask to the weight-gradient GEMM's
 *    operand); a plan is costly and is meant to be reused across many
 *    executes.
 *  - Fusing bias addition with matrix multiplication using nvmath-python:
 *    Y = ReLU(WX + B); RELU_AUX_BIAS also writes an auxiliary output for the
 *    backward pass; planning is blocking and chooses the kernel; a plan must
 *    be freed; operands must live on one device with compatible dtypes or
 *    the call fails.
 *  - PyTorch inference cuBLASLt bias-fusion optimization: the epilogue
 *    attribute and the bias pointer are bound on the matmul descriptor, the
 *    compute type is 32-bit float.
 *  - ops-nn MatMul fusion (codearts), "Why MatMul is the inference
 *    bottleneck": with one token per step the product is bound by reading the
 *    weights, which selects the weight-streaming GEMV path below.
 *
 * Canonical form. D[m,n] = act(sum_k A[m,k] * B[k,n] + bias[m]) for
 * 0 <= m < M, 0 <= n < N; bias is broadcast over the columns n. For an
 * nn.Linear layer Y[T,out] = X[T,in] W[out,in]^T + b this is M = out,
 * N = T, K = in, A = W (K-major), B = X^T (X read as a K-major B), and D
 * stored column-major, which is Y[T,out] row-major.
 *
 * Ownership and threading. The caller owns every device buffer (A, B, bias,
 * D, aux, and the DRELU_BGRAD outputs). A plan owns its host state and a
 * device workspace allocated by ge_plan_create on the device current at
 * that time (an error word; for DRELU_BGRAD / DGELU_BGRAD and
 * DW_DRELU_BGRAD the reduction partials and counters; for DW_DRELU_BGRAD
 * run as two launches the dZ buffer, K x lda elements; for the norm
 * epilogues the per-token statistics; for a split-K tail its fp32 pieces;
 * for stream-K tiles the workers' fp32 pieces and the flags that order
 * them).
 * ge_execute never allocates and only enqueues work on the given stream;
 * the caller synchronises. Executes of one plan must be ordered on one
 * stream: two executes of the same plan that overlap on the GPU race on its
 * workspace. Distinct plans are independent, and plans may be created,
 * executed and freed from several host threads.
 *
 * Environment (read by ge_plan_create, for tuning sweeps; unset in normal
 * use): GE_TILE_N = 128 | 256 | 224 (224: 2-SM pairs, K-major B' only) and
 * GE_PAIR = 0 | 1 force the tensor-core tile;
 * GE_SPLIT_TAIL = 0 disables the split-K tail; GE_EPI_WARPS = 4 | 8 forces the
 * epilogue width; GE_GROUP_M = g sets how many M-tiles the tile order sweeps
 * together; GE_DRELU_SPLITS = n sets the standalone D*_BGRAD row splits;
 * GE_KB = 64 forces one 64-wide k panel per pipeline stage (the default is
 * two, in one TMA box per operand, when K is a multiple of 128);
 * GE_STREAM_K = 1 shares the last waves' tiles out as stream-K k-ranges
 * whenever the last wave is ragged (default off); GE_DW_MASK = gemm selects
 * the in-GEMM form of DW_DRELU_BGRAD (default: two launches);
 * GE_TWO_PRODUCERS = 0 | 1 forces the tensor-core kernel's B loads onto the
 * stage's producer or a second producer warp (default: the second one when
 * an operand is M/N-major); for ge_execute_chain, GE_CHAIN_PRODUCERS = 1 |
 * 2 | 3 producer warps per block (default 3) and GE_CHAIN_INFLIGHT = n bulk
 * copies in flight per block (default half the ring).
 * They change speed, never results beyond rounding order.
 *
 * Errors. Every call returns a status and never aborts or prints. Arguments
 * are validated before anything is launched.
 */
#ifndef GE_H_
#define GE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ge_plan_s* ge_plan_t;

typedef enum {
  GE_OK = 0,
  GE_ERR_INVALID_ARG = 1,     /* null/negative/inconsistent argument           */
  GE_ERR_UNSUPPORTED = 2,     /* dtype / epilogue / layout not implemented     */
  GE_ERR_ALIGNMENT = 3,       /* pointer or leading dimension not 16-B aligned */
  GE_ERR_DEVICE_MISMATCH = 4, /* a buffer is not on the plan's device          */
  GE_ERR_CUDA = 5,            /* a CUDA runtime call or a launch failed        */
  GE_ERR_TIMEOUT = 6,         /* a bounded device-side wait expired            */
  GE_ERR_OOM = 7,             /* plan workspace allocation failed              */
  GE_ERR_DEVICE_CHECK = 8     /* a device-side index, offset or mbarrier-phase
                                 check of a debug build (GE_DEBUG) failed      */
} ge_status_t;

/* Epilogues (nvmath-python MatmulEpilog names). NONE is D = A.B. */
typedef enum {
  GE_EPI_NONE = 0,
  GE_EPI_BIAS = 1,          /* D = A.B + bias                                  */
  GE_EPI_RELU_BIAS = 2,     /* D = max(A.B + bias, 0)                          */
  GE_EPI_GELU_BIAS = 3,     /* D = gelu_tanh(A.B + bias)                       */
  GE_EPI_RELU_AUX_BIAS = 4, /* RELU_BIAS plus the bit-packed mask (z > 0)      */
  GE_EPI_DRELU_BGRAD = 5,   /* backward: dZ = dY * mask, bgrad = sum_n dZ      */
  GE_EPI_GELU_ERF_BIAS = 6, /* D = z * Phi(z), z = A.B + bias (exact erf GELU) */
  GE_EPI_GELU_AUX_BIAS = 7, /* GELU_BIAS plus z = A.B + bias kept as aux       */
  GE_EPI_DGELU_BGRAD = 8,   /* backward: dZ = dY * gelu'(z), bgrad = sum_n     */
  /* MatMul + bias + residual + norm over the M features (ge_execute_norm): */
  GE_EPI_BIAS_RESIDUAL_RMSNORM = 9,
  GE_EPI_BIAS_RESIDUAL_LAYERNORM = 10,
  /* weight gradient of a RELU_AUX_BIAS layer, the ReLU backward applied to
   * the A operand (dY) as it is loaded; bgrad from the same pass:          */
  GE_EPI_DW_DRELU_BGRAD = 11
} ge_epilogue_t;

/* GE_BF16: bfloat16 (1 sign, 8 exponent, 7 fraction bits), the other 16-bit
 * operand type of the tensor cores' f16 kind. */
typedef enum { GE_F16 = 0, GE_F32 = 1, GE_BF16 = 2 } ge_dtype_t;

/* Operand storage. A: K_MAJOR -> A[m,k] at A[m*lda + k]; MN_MAJOR -> A[k*lda + m].
 *                  B: K_MAJOR -> B[k,n] at B[n*ldb + k]; MN_MAJOR -> B[k*ldb + n]. */
typedef enum { GE_K_MAJOR = 0, GE_MN_MAJOR = 1 } ge_major_t;

/* D storage: ROW -> D[m,n] at D[m*ldd + n]; COL -> D[m,n] at D[n*ldd + m]. */
typedef enum { GE_D_ROW = 0, GE_D_COL = 1 } ge_dlayout_t;

/* Leading dimensions in elements (ld_aux of a mask in 32-bit words, of the
 * GELU_AUX_BIAS / DGELU_BGRAD pre-activation in elements); 0 selects the
 * packed default (K or M/N for the operands, the contiguous extent of D,
 * ceil(len/128)*4 words for the mask, and the contiguous extent of D rounded
 * up to 8 for the pre-activation). Every leading dimension must be a
 * multiple of 8 elements (16 bytes), a mask's ld_aux a multiple of 4 words. */
typedef struct {
  ge_major_t a;
  ge_major_t b;
  ge_dlayout_t d;
  int64_t lda, ldb, ldd, ld_aux;
} ge_layout_t;

/* Kernel path a plan selected (for inspection and benchmarks). */
typedef enum {
  GE_PATH_TC_GEMM = 0,   /* tcgen05 tensor-core GEMM with fused epilogue      */
  GE_PATH_GEMV = 1,      /* weight-streaming GEMV, N <= 4 (up to 16 when D's
                            stride is not a multiple of 8)                   */
  GE_PATH_DRELU = 2      /* DRELU_BGRAD streaming reduction                   */
} ge_path_t;

/*
 * ge_plan_create: validate a problem and choose its kernel.
 *   out      : receives the plan (set to NULL on failure).
 *   M, N, K  : problem size. M, N >= 1. K >= 1 for the forward epilogues;
 *              with DRELU_BGRAD or DGELU_BGRAD, K == 0 selects the standalone
 *              kernel on a stored dY and K >= 1 the GEMM-epilogue form (the
 *              gradient factor is applied to the product A.B). M, N, K < 2^31.
 *   a, b, d  : operand and output dtypes: all GE_F16 or all GE_BF16. The
 *              bias (and the standalone DRELU_BGRAD's dY and dZ) has the
 *              same type; the DRELU_BGRAD bias gradient stays fp32.
 *   compute  : accumulation dtype; GE_F32 only.
 *   epi      : epilogue.
 *   layout   : may be NULL = {A K_MAJOR, B MN_MAJOR, D ROW, packed lds}.
 * The device current at this call owns the plan's workspace; every execute
 * must pass buffers that live on that device. Leading dimensions must be
 * multiples of 8 elements on the tensor-core path (every operand and D), and
 * for lda/ldb on the GEMV path; ldd for DRELU_BGRAD.
 * Returns GE_OK, GE_ERR_INVALID_ARG, GE_ERR_UNSUPPORTED, GE_ERR_ALIGNMENT,
 * GE_ERR_CUDA (no device) or GE_ERR_OOM.
 */
ge_status_t ge_plan_create(ge_plan_t* out, int64_t M, int64_t N, int64_t K,
                           ge_dtype_t a, ge_dtype_t b, ge_dtype_t d,
                           ge_dtype_t compute, ge_epilogue_t epi,
                           const ge_layout_t* layout);

/*
 * ge_execute: enqueue the planned operation on `stream` (a cudaStream_t;
 * NULL = the legacy default stream). All pointers are device pointers of
 * the plan's device (alignment rules at the end of this comment).
 * Forward epilogues:
 * (T below is the plan's element type, fp16 or bf16.)
 *   A, B  : T operands in the planned layouts (read only).
 *   bias  : T [M] (read only); required for every *_BIAS epilogue,
 *           ignored for NONE.
 *   D     : T output, written once.
 *   aux   : RELU_AUX_BIAS only: uint32 mask words, ge_aux_bytes(plan) bytes.
 *           Bit (c % 32) of word aux[r*ld_aux + c/32] is 1 iff the fp32
 *           pre-activation of the element at stored row r, contiguous index c
 *           of D is > 0 ((r,c) = (m,n) for D ROW, (n,m) for D COL). Words up
 *           to ceil(len/128)*4 of each row are written; bits past the end of
 *           the row are 0.
 *   aux   : GELU_AUX_BIAS: T [rows of D][ld_aux] (ge_aux_bytes(plan) bytes,
 *           16-byte aligned), stored like D: z = A.B + bias rounded once to T
 *           (the pre-activation DGELU_BGRAD differentiates at).
 * DRELU_BGRAD as a GEMM epilogue (K >= 1): the backward product dH = A.B
 * (fp32 accumulate) is masked before its single store:
 *   A, B  : T operands as for the forward epilogues.
 *   aux   : the forward mask (read only), same packing as RELU_AUX_BIAS.
 *   D     : dZ, T: dZ[m,n] = T(dH[m,n]) where the bit is set, else +0.
 *   bias  : OUTPUT, fp32 [M]: bgrad[m] = sum over n of the masked fp32 dH,
 *           reduced in a fixed order (per-tile partial sums in the plan
 *           workspace, then one ordered pass), 16-byte aligned.
 * DGELU_BGRAD (tanh-GELU backward; GELU counterpart of DRELU_BGRAD): as
 * DRELU_BGRAD in both forms, with aux = the forward's z (T, stored like D,
 * ld_aux elements, 16-byte aligned, read only) in place of the mask:
 *   dZ[m,n] = T(g[m,n]), g = (dH or dY)[m,n] * gelu'(z[m,n]) in fp32, where
 *   gelu'(z) = 0.5 (1 + t) + 0.5 z (1 - t^2) sqrt(2/pi) (1 + 0.134145 z^2),
 *   t = tanh(sqrt(2/pi) (z + 0.044715 z^3)); bgrad[m] = sum over n of the
 *   unrounded fp32 g, in a fixed order. dZ may alias dY, not aux.
 * DW_DRELU_BGRAD (weight gradient of a RELU_AUX_BIAS layer whose forward D
 * was column-major, Y[tokens][features], with the ReLU backward applied to
 * the A operand. Plan: M = features, N = the other operand's width, K =
 * tokens; layout a = MN_MAJOR, d = ROW; ld_aux in words, default
 * ceil(M/128)*4). By default it runs as two launches, the standalone
 * DRELU_BGRAD pass storing dZ = dY * mask in a buffer the plan holds
 * (K x lda elements) and the NONE GEMM on it; with GE_DW_MASK = gemm in the
 * environment at plan creation the mask is applied inside the GEMM as it
 * loads the operand (dZ never stored; four more warps mask each stage in
 * shared memory). Both give the same dW and bias gradient:
 *   A     : dY, T [K tokens][lda >= M] (read only).
 *   B     : T operand in the planned layout (X: MN_MAJOR [K][ldb >= N]).
 *   aux   : the forward mask (read only), [K][ld_aux] uint32 words packed
 *           along the M features (the RELU_AUX_BIAS packing of a column-major
 *           forward D), 16-byte aligned.
 *   D     : dW, T: D[m,n] = T(sum over k of dZ[k,m] * B[k,n]) in fp32, with
 *           dZ[k,m] = dY[k,m] where bit (m % 32) of aux[k*ld_aux + m/32] is
 *           set, else +0.
 *   bias  : OUTPUT, fp32 [M] or NULL (not wanted): bgrad[m] = sum over k of
 *           dZ[k,m], in fp32 in a fixed order, 16-byte aligned.
 *   A, B, D and aux 16-byte aligned; the tensor-core path only. (The
 *   in-GEMM form measured 1.74 ms at 11008 x 4096 x 8192 against 0.46 ms
 *   for the two launches: it saves the dZ round trip through HBM but adds a
 *   shared-memory pass per operand stage and a hand-off to the MMA.)
 * DRELU_BGRAD standalone (K == 0; dY and dZ are [M,N] in the planned D layout):
 *   A     : dY, T (read only).           B : unused (may be NULL).
 *   aux   : the forward mask (read only). D : dZ, T; may alias A.
 *   bias  : OUTPUT, fp32 [M]: bgrad[m] = sum over n of dZ[m,n], reduced in
 *           fp32 in a fixed order (deterministic run to run).
 *   dZ[m,n] = dY[m,n] where the mask bit is set, +0 elsewhere.
 * Returns GE_OK, GE_ERR_INVALID_ARG (null plan or a required pointer null),
 * GE_ERR_ALIGNMENT, GE_ERR_DEVICE_MISMATCH (a pointer that is not device
 * memory of the plan's device) or GE_ERR_CUDA (launch failure). A device-side
 * wait that expires during the kernel is reported by
 * ge_get_last_device_error, not here (execute does not synchronise).
 * Pointer alignment: A, B (and D on the tensor-core path) 16 bytes; bias 2;
 * aux 4 (16 for DRELU_BGRAD, where A, D and the fp32 bias output are 16).
 */
ge_status_t ge_execute(ge_plan_t plan, const void* A, const void* B,
                       const void* bias, void* D, void* aux, void* stream);

/*
 * ge_execute_unfused: the three-kernel baseline on the same inputs: the
 * plan's GEMM with no epilogue writes D, then one kernel reads D, adds the
 * bias and writes D, then one kernel reads D, applies the activation (and
 * writes the mask for RELU_AUX_BIAS, from the rounded z) and writes D
 * (ops-nn MatMul fusion, "ops-nn's MatMul fusion strategy", the unfused
 * three-step flow). Only for BIAS / RELU_BIAS / GELU_BIAS / RELU_AUX_BIAS /
 * GELU_ERF_BIAS / GELU_AUX_BIAS plans. Arguments and errors as ge_execute.
 */
ge_status_t ge_execute_unfused(ge_plan_t plan, const void* A, const void* B,
                               const void* bias, void* D, void* aux,
                               void* stream);

/*
 * ge_execute_norm: MatMul + bias + residual + normalisation, the structural
 * fusion of ops-nn MatMul fusion (codearts), "ops-nn's MatMul fusion
 * strategy", second level (MatMul + LayerNorm / RMSNorm with the residual
 * connection; the norm reduces across the channel dimension). For a plan
 * created with GE_EPI_BIAS_RESIDUAL_RMSNORM or _LAYERNORM and a column-major
 * D (D[m,n] at n*ldd + m: N tokens of M contiguous features; other layouts
 * are GE_ERR_UNSUPPORTED at planning):
 *   h[m,n] = sum_k A[m,k] B[k,n] + bias[m] + residual[m,n]   (fp32)
 *   H      = h rounded to T (the new residual stream), stored like D
 *   for every token n, over its M features (population statistics):
 *     RMSNorm:   Y = h * rsqrt(mean(h^2) + eps) * gamma
 *     LayerNorm: Y = (h - mu) * rsqrt(mean((h - mu)^2) + eps) * gamma + beta
 *   Y is stored like D, rounded to T.
 * The GEMM (or, for N <= 16, the GEMV) adds bias and residual in its
 * epilogue and stores H once; one more pass reads each token's row of H
 * once and writes Y (the statistics are taken from the stored H).
 *   A, B              : T operands in the planned layouts (read only).
 *   bias, gamma, beta : T [M] (read only); beta only for LayerNorm (may be
 *                       NULL for RMSNorm). gamma, beta 16-byte aligned.
 *   residual, H, Y    : T, laid out like D (ldd), 16-byte aligned. H may be
 *                       the residual buffer (in-place update of the residual
 *                       stream); Y may be H.
 *   eps               : >= 0, added to the mean square / variance.
 * Returns GE_OK, GE_ERR_UNSUPPORTED (not a norm plan), GE_ERR_INVALID_ARG,
 * GE_ERR_ALIGNMENT, GE_ERR_DEVICE_MISMATCH or GE_ERR_CUDA. ge_execute on a
 * norm plan returns GE_ERR_UNSUPPORTED.
 */
ge_status_t ge_execute_norm(ge_plan_t plan, const void* A, const void* B, const void* bias,
                            const void* residual, const void* gamma, const void* beta,
                            void* H, void* Y, float eps, void* stream);

/*
 * ge_execute_norm_unfused: the same result by separate kernels, the flow the
 * fusion replaces: the GEMM writes A.B as H, then bias add, residual add and
 * the norm pass each read and write H. H must not be the residual buffer.
 */
ge_status_t ge_execute_norm_unfused(ge_plan_t plan, const void* A, const void* B,
                                    const void* bias, const void* residual,
                                    const void* gamma, const void* beta, void* H, void* Y,
                                    float eps, void* stream);

/*
 * ge_execute_chain: a stack of decode projections in one launch (ops-nn
 * MatMul fusion (codearts), "Why MatMul is the inference bottleneck": a
 * decode step carries one token's activations through one weight matrix
 * after another, and each costs the time to read its weights once from HBM).
 * For a decode-sized plan (N <= 16, A and B K-major; whichever path its own
 * ge_execute takes) that is
 * square (M == K) with a column-major D (N rows of M features, the layout of
 * the next layer's K-major B), and an epilogue in NONE / BIAS / RELU_BIAS /
 * GELU_BIAS / GELU_ERF_BIAS:
 *   Y_0 = act(A_0 . X + bias_0),   Y_l = act(A_l . Y_(l-1) + bias_l),
 * every Y_l rounded to T and stored, and layer l reading exactly the stored
 * Y_(l-1).
 *   layers : 1 .. 64.
 *   A      : host array of `layers` device pointers, T [M][lda] each (the
 *            plan's A layout), 16-byte aligned (read only).
 *   bias   : host array of `layers` device pointers, T [M] each, 2-byte
 *            aligned (read only); may be NULL for NONE.
 *   X      : T, N rows of K with the plan's ldb (read only), 16-byte aligned.
 *   Y      : T, layer l's output at Y + l * N * ldd elements, N rows of M with
 *            the plan's ldd; 16-byte aligned. Must not overlap X or weights.
 * K, ldb and ldd must be multiples of 8. One cooperative launch runs every
 * layer: each SM keeps its next weight rows -- of this layer and the
 * following ones -- streaming into shared memory while the grid waits for
 * the previous layer's outputs, which pass between the SMs as tagged words
 * in the plan's workspace (2 x N x M x 4 bytes, allocated by ge_plan_create
 * for every plan of this form). The launch needs every SM of the device
 * free of other work to start. Executes of one plan must be ordered on one
 * stream (they share the plan's synchronisation and exchange words).
 * Returns GE_OK, GE_ERR_UNSUPPORTED (plan not of this form, or the N
 * activation rows and one weight row segment do not fit in shared memory
 * together: K above about 77,000 for one token, 25,800 for four, 6,800
 * for 16),
 * GE_ERR_INVALID_ARG (layers out of range, a required pointer NULL),
 * GE_ERR_ALIGNMENT, GE_ERR_DEVICE_MISMATCH or GE_ERR_CUDA. Device waits are
 * bounded; an expired wait is reported by ge_get_last_device_error.
 */
ge_status_t ge_execute_chain(ge_plan_t plan, int64_t layers, const void* const* A,
                             const void* const* bias, const void* X, void* Y, void* stream);

/* Plan attributes (ge_plan_set_attr). */
typedef enum {
  /* value 1: A is never written by work queued earlier on the execute's
   * stream (model weights). Decode-sized plans (GE_PATH_GEMV) then launch
   * with programmatic dependent launch: the kernel may start while the
   * previous kernel on the stream is still running, streams its first weight
   * rows into shared memory, and only then waits for that kernel to finish
   * before it reads B (the activations) or writes D. Chains of decode
   * projections overlap one layer's weight fetch with the previous layer's
   * tail. Value 0 (default): the kernel starts after earlier work. Other
   * paths ignore the attribute. */
  GE_ATTR_STATIC_A = 0
} ge_plan_attr_t;

/* Set a plan attribute. Returns GE_OK, or GE_ERR_INVALID_ARG for a NULL
 * plan, an unknown attribute or a value outside its range. */
ge_status_t ge_plan_set_attr(ge_plan_t plan, ge_plan_attr_t attr, int64_t value);

/*
 * ge_plan_autotune: choose the plan's kernel configuration by timing.
 * Planning picks a configuration from the problem's shape; this call instead
 * runs every candidate of the tensor-core path (128-, 256- or (2-SM pairs,
 * K-major B') 224-column tiles, single-CTA or 2-SM pair tiles, with and
 * without the split-K tail or the stream-K last waves, pipeline stages of
 * one or two 64-wide k panels) `reps` times on the caller's buffers
 * (same meaning as ge_execute), keeps the fastest for every later execute,
 * and finishes with one execute in that configuration, so D / aux / bias
 * hold its results. It blocks the host until
 * the timing runs finish and may re-allocate the plan's tail workspace.
 * Plans of the other paths are left unchanged (GE_OK). Norm plans
 * (GE_EPI_BIAS_RESIDUAL_*) are not tuned: ge_execute does not run them, so
 * the call returns GE_ERR_UNSUPPORTED and the plan keeps its configuration.
 * reps in 1..1000.
 * The choice is also remembered for the process (per device, M, N, K,
 * epilogue, element type and layout): plans created later for the same
 * problem start from it (unless GE_TILE_N / GE_PAIR / GE_SPLIT_TAIL /
 * GE_STREAM_K are set in the environment).
 * Returns GE_OK or the first failing status (the plan then keeps a valid
 * configuration).
 */
ge_status_t ge_plan_autotune(ge_plan_t plan, const void* A, const void* B,
                             const void* bias, void* D, void* aux, void* stream,
                             int reps);

/* Forget every configuration remembered by ge_plan_autotune (existing plans
 * keep theirs). */
void ge_autotune_cache_clear(void);

/* The plan's tensor-core configuration: tile width, 2-SM pair mode (0: one
 * CTA per 128-row tile; 1: CTA pairs on 256-row tiles) and split-K pieces of the tail
 * (1 = none); zeros for other paths. Any pointer may be NULL. Returns the
 * path, or -1 for a NULL plan. */
int ge_plan_config(ge_plan_t plan, int* block_n, int* pair, int* split);

/* Stream-K (tensor-core path). When the last wave of output tiles would
 * leave workers (SMs, or SM pairs) idle, the planner may give the last
 * `n` tiles' k-block iterations out in equal contiguous ranges, one per
 * worker; a tile cut between workers is finished inside the GEMM by the
 * worker whose range starts it, which adds the others' fp32 pieces in k
 * order (bounded waits on flags in the plan workspace; an expired one
 * reports GE_ERR_TIMEOUT through ge_get_last_device_error). Every worker of
 * the launch has to be resident at once: the grid is the number that fits.
 * Returns n (0: none, or not a tensor-core plan), or -1 for a NULL plan. */
int ge_plan_stream_k_tiles(ge_plan_t plan);

/* Release the plan and its device workspace (NULL is accepted). The caller
 * must make sure no execute of the plan is still running on the GPU. */
ge_status_t ge_plan_free(ge_plan_t plan);

/* Bytes of aux output the caller allocates: the mask of RELU_AUX_BIAS or
 * the pre-activation of GELU_AUX_BIAS (0 otherwise). */
size_t ge_aux_bytes(ge_plan_t plan);

/* Row pitch of aux chosen by the plan: 32-bit words for a mask, elements for
 * a pre-activation (GELU_AUX_BIAS, DGELU_BGRAD); 0 if the plan has no aux. */
int64_t ge_aux_ld(ge_plan_t plan);

/* The kernel path the plan selected, or -1 for a NULL plan. */
int ge_plan_path(ge_plan_t plan);

/* Output-tile width (columns of one CTA tile, 0 if not a GEMM path). */
int ge_plan_tile_n(ge_plan_t plan);

/*
 * Read and clear the plan's device error word. Synchronises the device.
 * Returns GE_OK when no device-side wait of this plan has expired since the
 * last read, GE_ERR_TIMEOUT when one has (the kernel then stopped early and
 * its outputs are undefined), GE_ERR_DEVICE_CHECK when a check of a debug
 * build (compiled with GE_DEBUG) failed (the access was skipped; outputs
 * undefined), GE_ERR_CUDA if the read itself failed.
 */
ge_status_t ge_get_last_device_error(ge_plan_t plan);

/* Static description of a status code; never NULL. */
const char* ge_status_string(ge_status_t s);

/*
 * Test hook for the bounded-wait path: launches one CTA that waits on a
 * shared-memory barrier nobody arrives at, with a budget of `budget_cycles`
 * SM clock cycles (1 .. 2^31), then records the expiry in the plan's error
 * word and returns. The GPU context stays usable. Returns the launch status;
 * read the outcome with ge_get_last_device_error.
 */
ge_status_t ge_debug_wait_timeout(ge_plan_t plan, int64_t budget_cycles,
                                  void* stream);

/*
 * ge_drelu_bgrad_static: DRELU_BGRAD that allocates nothing.
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory: a framework whose caching allocator owns
 * all of it, a serving loop that must never block on cudaMalloc's implicit
 * device synchronisation, or a process held to a fixed memory budget where a
 * new allocation may fail. A plan needs cudaMalloc for its workspace, so this
 * entry point takes the problem directly and keeps its reduction scratch in
 * a fixed file-scope device array of GE_STATIC_SCRATCH_BYTES (4 MiB), which
 * every GPU that loads the library holds until the process exits.
 *   M, N, d, ldd, ld_aux : as a DRELU_BGRAD plan (K = 0) with layout d
 *                          (0 for ldd / ld_aux selects the packed default).
 *   dY, aux, dZ          : fp16 dY, uint32 mask, fp16 dZ (may alias dY),
 *                          device pointers, 16-byte aligned.
 *   bgrad                : OUTPUT fp32 [M], 16-byte aligned.
 *   stream               : cudaStream_t (NULL = legacy default stream).
 * Results are the same as the plan-based execute (the fp32 reduction may use
 * fewer row splits when the scratch is short, so bgrad can differ in the
 * last bits). The first call on each device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture. Every call shares the array and it keeps
 * the last call's contents: the call clears the counters it needs on
 * `stream` itself, and calls that overlap on the GPU race on the scratch, so
 * order them on one stream. Allocates nothing: no cudaMalloc, cudaFree or
 * allocating library routine.
 * Limit: for d == GE_D_COL, ceil(M/256)*4 bytes rounded up to 256 plus M*4
 * bytes must fit in GE_STATIC_SCRATCH_BYTES (M up to about one million);
 * larger problems return GE_ERR_UNSUPPORTED. d == GE_D_ROW uses no scratch.
 * Returns GE_OK, GE_ERR_INVALID_ARG, GE_ERR_ALIGNMENT, GE_ERR_UNSUPPORTED,
 * GE_ERR_DEVICE_MISMATCH (a pointer that is not memory of the current
 * device) or GE_ERR_CUDA.
 */
#define GE_STATIC_SCRATCH_BYTES ((size_t)4 << 20)
ge_status_t ge_drelu_bgrad_static(int64_t M, int64_t N, ge_dlayout_t d,
                                  int64_t ldd, int64_t ld_aux, const void* dY,
                                  const void* aux, void* dZ, void* bgrad,
                                  void* stream);

/* 1 if this library was compiled with the device-side checks (GE_DEBUG),
 * else 0. */
int ge_debug_checks(void);

/*
 * Test hook for the checking build: launches one thread whose GE_DEBUG
 * check fails by construction (it guards no memory access). In a build with
 * the checks, ge_get_last_device_error then returns GE_ERR_DEVICE_CHECK; in
 * the normal build the kernel does nothing and it returns GE_OK. Returns
 * the launch status.
 */
ge_status_t ge_debug_check_probe(ge_plan_t plan, void* stream);

/* Library version, "major.minor.patch". */
const char* ge_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GE_H_ */
