"""Python wrapper of the plain CPU oracle (``ge_oracle.cpp``).

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke``
and by the CPU-baseline leg of ``bench.py``; never by the library itself. It
imports nothing from the CUDA package and shares no code with it.

Arrays are numpy: fp16 operands are passed as their uint16 bit patterns, so
the oracle and the GPU see identical bits. Layout vocabulary (the oracle's
own; it mirrors the library's documented layouts):

* ``a_major``: ``"k"`` -> A[m,k] at ``A[m*lda + k]``; ``"m"`` -> ``A[k*lda + m]``
* ``b_major``: ``"k"`` -> B[k,n] at ``B[n*ldb + k]``; ``"n"`` -> ``B[k*ldb + n]``
* ``d_layout``: ``"row"`` -> D[m,n] at ``D[m*ldd + n]``; ``"col"`` -> ``D[n*ldd + m]``

What is computed, and the pages each step follows, is documented in
``ge_oracle.cpp``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ge_oracle.cpp")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libge_oracle.so")

EPILOGUES = {"none": 0, "bias": 1, "relu_bias": 2, "gelu_bias": 3, "relu_aux_bias": 4,
             "gelu_erf_bias": 6, "gelu_aux_bias": 7}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (plain -O2, no fast-math, no FP contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            lib.ora_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.ora_f16_to_f64.restype = ctypes.c_double
            lib.ora_f64_to_f16.argtypes = [ctypes.c_double]
            lib.ora_f64_to_f16.restype = ctypes.c_uint16
            lib.ora_act_f64.argtypes = [i32, ctypes.c_double]
            lib.ora_act_f64.restype = ctypes.c_double
            lib.ora_bf16_to_f64_array.argtypes = [vp, vp, i64]
            lib.ora_bf16_to_f64_array.restype = None
            lib.ora_f64_to_bf16_array.argtypes = [vp, vp, i64]
            lib.ora_f64_to_bf16_array.restype = None
            lib.ora_linear_forward_dt.argtypes = [i32, i64, i64, i64, vp, i32, i64, vp, i32, i64,
                                                  vp, i32, vp, i32, i64, vp, i64, vp, i32]
            lib.ora_linear_forward_dt.restype = i32
            lib.ora_drelu_bgrad_dt.argtypes = [i32, i64, i64, vp, i32, i64, vp, i64, vp, vp]
            lib.ora_drelu_bgrad_dt.restype = i32
            lib.ora_gemm_drelu_bgrad_dt.argtypes = [i32, i64, i64, i64, vp, i32, i64, vp, i32, i64, vp,
                                                    i64, vp, i32, i64, vp, i32]
            lib.ora_gemm_drelu_bgrad_dt.restype = i32
            lib.ora_f16_to_f64_array.argtypes = [vp, vp, i64]
            lib.ora_f16_to_f64_array.restype = None
            lib.ora_f64_to_f16_array.argtypes = [vp, vp, i64]
            lib.ora_f64_to_f16_array.restype = None
            lib.ora_linear_forward.argtypes = [i64, i64, i64, vp, i32, i64, vp, i32, i64,
                                               vp, i32, vp, i32, i64, vp, i64, vp, i32]
            lib.ora_linear_forward.restype = i32
            lib.ora_gemm_drelu_bgrad.argtypes = [i64, i64, i64, vp, i32, i64, vp, i32, i64, vp, i64,
                                                 vp, i32, i64, vp, i32]
            lib.ora_gemm_drelu_bgrad.restype = i32
            lib.ora_drelu_bgrad.argtypes = [i64, i64, vp, i32, i64, vp, i64, vp, vp]
            lib.ora_drelu_bgrad.restype = i32
            lib.ora_gelu_aux_forward_dt.argtypes = [i32, i64, i64, i64, vp, i32, i64, vp, i32, i64,
                                                    vp, vp, i32, i64, vp, i64, vp, i32]
            lib.ora_gelu_aux_forward_dt.restype = i32
            lib.ora_gelu_grad_f64.argtypes = [ctypes.c_double]
            lib.ora_gelu_grad_f64.restype = ctypes.c_double
            lib.ora_dgelu_bgrad_dt.argtypes = [i32, i64, i64, vp, i32, i64, vp, i64, vp, vp]
            lib.ora_dgelu_bgrad_dt.restype = i32
            lib.ora_gemm_dgelu_bgrad_dt.argtypes = [i32, i64, i64, i64, vp, i32, i64, vp, i32, i64, vp,
                                                    i64, vp, i32, i64, vp, i32]
            lib.ora_gemm_dgelu_bgrad_dt.restype = i32
            lib.ora_linear_norm_dt.argtypes = [i32, i32, i64, i64, i64, vp, i32, i64, vp, i32, i64, vp, vp,
                                               vp, vp, ctypes.c_double, vp, vp, i32, i64, i32]
            lib.ora_linear_norm_dt.restype = i32
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


DTYPES = {"f16": 0, "bf16": 1}


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


def default_ld_aux(contiguous_len: int) -> int:
    """Mask row pitch in 32-bit words: one bit per element of a stored row of
    D, rows padded to a multiple of 16 bytes (4 words)."""
    return ((contiguous_len + 127) // 128) * 4


def f16_decode(bits, dtype: str = "f16") -> np.ndarray:
    """Bit patterns of fp16 (or, with dtype="bf16", bfloat16) values -> fp64."""
    lib = _load()
    bits = _u16(bits)
    out = np.empty(bits.shape, np.float64)
    fn = lib.ora_f16_to_f64_array if dtype == "f16" else lib.ora_bf16_to_f64_array
    fn(_ptr(bits), _ptr(out), bits.size)
    return out


def bf16_decode(bits) -> np.ndarray:
    return f16_decode(bits, "bf16")


def bf16_encode(x) -> np.ndarray:
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint16)
    lib.ora_f64_to_bf16_array(_ptr(x), _ptr(out), x.size)
    return out


def act_f64(epilogue: str, z: float) -> float:
    """The epilogue's activation applied to one fp64 value (no rounding)."""
    return float(_load().ora_act_f64(EPILOGUES[epilogue], float(z)))


def f16_encode(x) -> np.ndarray:
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint16)
    lib.ora_f64_to_f16_array(_ptr(x), _ptr(out), x.size)
    return out


def linear_forward(A, B, bias, epilogue: str, M: int, N: int, K: int, *,
                   a_major: str = "k", b_major: str = "k", d_layout: str = "row",
                   lda: int | None = None, ldb: int | None = None,
                   ldd: int | None = None, ld_aux: int | None = None,
                   threads: int | None = None, dtype: str = "f16",
                   ld_zaux: int | None = None) -> dict:
    """D = act(A.B + bias) in fp64, rounded once to fp16 (or bfloat16 with
    dtype="bf16"; A, B, bias and D all of that type).

    Returns ``{"D": uint16 bits, "Z": fp64 pre-activation, "aux": uint32 mask
    words or None}``; D and Z are flat arrays of ``rows*ldd`` elements in the
    stored layout, aux is ``rows*ld_aux`` words. For "gelu_aux_bias" the
    result also holds ``"zaux"``: z rounded to the element type, ``rows *
    ld_zaux`` elements stored like D (ld_zaux defaults to the contiguous
    length rounded up to 8).
    """
    lib = _load()
    epi = EPILOGUES[epilogue]
    if lda is None:
        lda = K if a_major == "k" else M
    if ldb is None:
        ldb = K if b_major == "k" else N
    rows, cols = (M, N) if d_layout == "row" else (N, M)
    if ldd is None:
        ldd = cols
    if ld_aux is None:
        ld_aux = default_ld_aux(cols)
    A = _u16(A)
    B = _u16(B)
    bias = None if bias is None else _u16(bias)
    D = np.zeros(rows * ldd, np.uint16)
    Z = np.zeros(rows * ldd, np.float64)
    aux = np.zeros(rows * ld_aux, np.uint32) if epilogue == "relu_aux_bias" else None
    if threads is None:
        threads = os.cpu_count() or 1
    if epilogue == "gelu_aux_bias":
        ld_zaux = ld_zaux or default_ld_zaux(cols)
        zaux = np.zeros(rows * ld_zaux, np.uint16)
        rc = lib.ora_gelu_aux_forward_dt(DTYPES[dtype], M, N, K, _ptr(A), 0 if a_major == "k" else 1,
                                         lda, _ptr(B), 0 if b_major == "k" else 1, ldb, _ptr(bias),
                                         _ptr(D), 0 if d_layout == "row" else 1, ldd, _ptr(zaux), ld_zaux,
                                         _ptr(Z), int(threads))
        if rc != 0:
            raise ValueError("oracle rejected the arguments")
        return {"D": D, "Z": Z, "aux": None, "zaux": zaux, "ldd": ldd, "ld_zaux": ld_zaux}
    rc = lib.ora_linear_forward_dt(DTYPES[dtype], M, N, K, _ptr(A), 0 if a_major == "k" else 1, lda,
                                   _ptr(B), 0 if b_major == "k" else 1, ldb,
                                   _ptr(bias), epi, _ptr(D), 0 if d_layout == "row" else 1, ldd,
                                   _ptr(aux), ld_aux, _ptr(Z), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return {"D": D, "Z": Z, "aux": aux, "ldd": ldd, "ld_aux": ld_aux}


def drelu_bgrad(dY, aux, M: int, N: int, *, d_layout: str = "row",
                ldd: int | None = None, ld_aux: int | None = None, dtype: str = "f16"):
    """Backward epilogue: dZ = dY where the mask bit is set else +0 (fp16 bits),
    bgrad[m] = sum over n of dZ[m,n] in fp64."""
    lib = _load()
    rows, cols = (M, N) if d_layout == "row" else (N, M)
    if ldd is None:
        ldd = cols
    if ld_aux is None:
        ld_aux = default_ld_aux(cols)
    dY = _u16(dY)
    aux = np.ascontiguousarray(aux, dtype=np.uint32)
    dZ = np.zeros(rows * ldd, np.uint16)
    bgrad = np.zeros(M, np.float64)
    rc = lib.ora_drelu_bgrad_dt(DTYPES[dtype], M, N, _ptr(dY), 0 if d_layout == "row" else 1, ldd,
                                _ptr(aux), ld_aux, _ptr(dZ), _ptr(bgrad))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return dZ, bgrad


def gemm_drelu_bgrad(A, B, aux, M: int, N: int, K: int, *, a_major: str = "k", b_major: str = "k",
                     d_layout: str = "row", lda: int | None = None, ldb: int | None = None,
                     ldd: int | None = None, ld_aux: int | None = None, threads: int | None = None,
                     dtype: str = "f16"):
    """DRELU_BGRAD applied to a product: dZ = fp16(A.B) where the mask bit is
    set else +0; bgrad[m] = sum over n of the unrounded masked product (fp64)."""
    lib = _load()
    if lda is None:
        lda = K if a_major == "k" else M
    if ldb is None:
        ldb = K if b_major == "k" else N
    rows, cols = (M, N) if d_layout == "row" else (N, M)
    if ldd is None:
        ldd = cols
    if ld_aux is None:
        ld_aux = default_ld_aux(cols)
    A = _u16(A)
    B = _u16(B)
    aux = np.ascontiguousarray(aux, dtype=np.uint32)
    dZ = np.zeros(rows * ldd, np.uint16)
    bgrad = np.zeros(M, np.float64)
    if threads is None:
        threads = os.cpu_count() or 1
    rc = lib.ora_gemm_drelu_bgrad_dt(DTYPES[dtype], M, N, K, _ptr(A), 0 if a_major == "k" else 1, lda,
                                     _ptr(B), 0 if b_major == "k" else 1, ldb, _ptr(aux), ld_aux, _ptr(dZ),
                                     0 if d_layout == "row" else 1, ldd, _ptr(bgrad), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return dZ, bgrad


def default_ld_zaux(contiguous_len: int) -> int:
    """Row pitch (elements) of a GELU_AUX_BIAS pre-activation output: the
    contiguous length rounded up to 8 elements (16 bytes)."""
    return (contiguous_len + 7) // 8 * 8


def gelu_grad_f64(z: float) -> float:
    """Derivative of the tanh-form GELU at z (fp64)."""
    return _load().ora_gelu_grad_f64(float(z))


def dw_drelu_bgrad(dY, aux, X, M: int, N: int, K: int, *, lda: int | None = None, ldb: int | None = None,
                   ld_aux: int | None = None, dtype: str = "f16"):
    """Weight gradient of a RELU_AUX_BIAS layer whose forward D was column-major
    (nvmath-python cuBLASLt bias-fusion guide, "Advanced techniques", backward
    item: the mask kept by the forward gates the incoming gradient). dY is
    stored [K tokens][lda >= M features] and the mask [K][ld_aux] words along
    the features. By definition, two pinned steps: dZ = dY where the mask bit
    is set else +0 and bgrad[m] = sum over the K tokens of dZ (``drelu_bgrad``
    on the column-major layout), then dW = dZ^T X (``linear_forward`` with no
    epilogue: A = dZ read M-major, B = X [K][ldb >= N] read N-major, D
    row-major [M][N]). Returns (dW bits, flat M*N; bgrad fp64 [M])."""
    lda = lda or M
    dZ, bgrad = drelu_bgrad(dY, aux, M, K, d_layout="col", ldd=lda, ld_aux=ld_aux, dtype=dtype)
    out = linear_forward(dZ, X, None, "none", M, N, K, a_major="m", b_major="n", d_layout="row", lda=lda,
                         ldb=ldb, dtype=dtype)
    return out["D"], bgrad


def dgelu_bgrad(dY, zaux, M: int, N: int, *, d_layout: str = "row", ldd: int | None = None,
                ld_zaux: int | None = None, dtype: str = "f16"):
    """Backward epilogue of GELU_AUX_BIAS: g = dY * gelu'(z) with z the stored
    (rounded) pre-activation; dZ = g rounded to the element type; bgrad[m] =
    sum over n of the unrounded g (fp64)."""
    lib = _load()
    rows, cols = (M, N) if d_layout == "row" else (N, M)
    ldd = ldd or cols
    ld_zaux = ld_zaux or default_ld_zaux(cols)
    dY = _u16(dY)
    zaux = _u16(zaux)
    dZ = np.zeros(rows * ldd, np.uint16)
    bgrad = np.zeros(M, np.float64)
    rc = lib.ora_dgelu_bgrad_dt(DTYPES[dtype], M, N, _ptr(dY), 0 if d_layout == "row" else 1, ldd,
                                _ptr(zaux), ld_zaux, _ptr(dZ), _ptr(bgrad))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return dZ, bgrad


def gemm_dgelu_bgrad(A, B, zaux, M: int, N: int, K: int, *, a_major: str = "k", b_major: str = "k",
                     d_layout: str = "row", lda: int | None = None, ldb: int | None = None,
                     ldd: int | None = None, ld_zaux: int | None = None, threads: int | None = None,
                     dtype: str = "f16"):
    """DGELU_BGRAD applied to a product dH = A.B: dZ = (dH * gelu'(z)) rounded;
    bgrad[m] = sum over n of the unrounded dH * gelu'(z) (fp64)."""
    lib = _load()
    lda = lda or (K if a_major == "k" else M)
    ldb = ldb or (K if b_major == "k" else N)
    rows, cols = (M, N) if d_layout == "row" else (N, M)
    ldd = ldd or cols
    ld_zaux = ld_zaux or default_ld_zaux(cols)
    A = _u16(A)
    B = _u16(B)
    zaux = _u16(zaux)
    dZ = np.zeros(rows * ldd, np.uint16)
    bgrad = np.zeros(M, np.float64)
    threads = threads or (os.cpu_count() or 1)
    rc = lib.ora_gemm_dgelu_bgrad_dt(DTYPES[dtype], M, N, K, _ptr(A), 0 if a_major == "k" else 1, lda,
                                     _ptr(B), 0 if b_major == "k" else 1, ldb, _ptr(zaux), ld_zaux,
                                     _ptr(dZ), 0 if d_layout == "row" else 1, ldd, _ptr(bgrad),
                                     int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return dZ, bgrad


NORMS = {"rmsnorm": 0, "layernorm": 1}


def linear_norm(A, B, bias, res, gamma, beta, norm: str, M: int, N: int, K: int, *, eps: float = 1e-5,
                a_major: str = "k", b_major: str = "k", d_layout: str = "col", lda: int | None = None,
                ldb: int | None = None, ldd: int | None = None, threads: int | None = None,
                dtype: str = "f16"):
    """MatMul + bias + residual, then RMSNorm / LayerNorm over the M output
    features of every token n. Returns (H, Y): the rounded h = A.B + bias +
    res and the rounded normalised output, both stored like D (flat uint16,
    rows * ldd)."""
    lib = _load()
    lda = lda or (K if a_major == "k" else M)
    ldb = ldb or (K if b_major == "k" else N)
    rows, cols = (M, N) if d_layout == "row" else (N, M)
    ldd = ldd or cols
    A, B, bias, res, gamma = _u16(A), _u16(B), _u16(bias), _u16(res), _u16(gamma)
    beta = None if beta is None else _u16(beta)
    H = np.zeros(rows * ldd, np.uint16)
    Y = np.zeros(rows * ldd, np.uint16)
    threads = threads or (os.cpu_count() or 1)
    rc = lib.ora_linear_norm_dt(DTYPES[dtype], NORMS[norm], M, N, K, _ptr(A), 0 if a_major == "k" else 1, lda,
                                _ptr(B), 0 if b_major == "k" else 1, ldb, _ptr(bias), _ptr(res), _ptr(gamma),
                                _ptr(beta), float(eps), _ptr(H), _ptr(Y), 0 if d_layout == "row" else 1, ldd,
                                int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return H, Y


def decode_chain(As, biases, X, epilogue: str, M: int, N: int, *, dtype: str = "f16",
                 threads: int | None = None):
    """A stack of decode projections, each layer's stored output the next
    layer's input (ops-nn MatMul fusion, "Why MatMul is the inference
    bottleneck": a decode step carries one token's activations through one
    weight matrix after another, each read once):

        Y_0 = act(A_0 . X + b_0),   Y_l = act(A_l . Y_(l-1) + b_l),

    every layer square (K = M) and computed by ``linear_forward`` (fp64,
    rounded once to the element type), so layer l reads exactly the rounded
    Y_(l-1). X is N tokens x M (a K-major B); each Y_l is stored like a
    column-major D, N rows of M. ``As`` and ``biases`` list the layers' bit
    patterns (a bias may be None for "none"). Returns the layers' outputs,
    flat uint16 arrays of N*M."""
    prev = _u16(X)
    outs = []
    for A, b in zip(As, biases):
        r = linear_forward(A, prev, b, epilogue, M, N, M, a_major="k", b_major="k", d_layout="col",
                           dtype=dtype, threads=threads)
        outs.append(r["D"])
        prev = r["D"]
    return outs
