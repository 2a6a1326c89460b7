"""Python binding of the GB300 fused linear-layer engine.

Argument marshalling only: every call forwards to the C ABI of
``_build/libgemm_epilogues.so`` (declared in ``include/ge.h``), with the same
names. Buffers are passed as raw device pointers; anything exposing
``data_ptr()`` (a torch tensor) or a plain integer is accepted. Streams are
``cudaStream_t`` handles: an integer, an object with ``cuda_stream`` (a torch
stream) or ``None`` for the legacy default stream.

There is no fallback: if the library has not been built, or cannot be loaded,
every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
# GE_DEBUG_LIB=1 selects the checking build (build.build(debug=True)): the
# same kernels compiled with GE_DEBUG, whose index, offset and mbarrier-phase
# checks report GE_ERR_DEVICE_CHECK through ge_get_last_device_error.
LIB_PATH = os.path.join(_HERE, "_build_debug" if os.environ.get("GE_DEBUG_LIB") == "1" else "_build",
                        "libgemm_epilogues.so")

# ge_status_t
GE_OK = 0
GE_ERR_INVALID_ARG = 1
GE_ERR_UNSUPPORTED = 2
GE_ERR_ALIGNMENT = 3
GE_ERR_DEVICE_MISMATCH = 4
GE_ERR_CUDA = 5
GE_ERR_TIMEOUT = 6
GE_ERR_OOM = 7
GE_ERR_DEVICE_CHECK = 8
# ge_epilogue_t
GE_EPI_NONE = 0
GE_EPI_BIAS = 1
GE_EPI_RELU_BIAS = 2
GE_EPI_GELU_BIAS = 3
GE_EPI_RELU_AUX_BIAS = 4
GE_EPI_DRELU_BGRAD = 5
GE_EPI_GELU_ERF_BIAS = 6
GE_EPI_GELU_AUX_BIAS = 7
GE_EPI_DGELU_BGRAD = 8
GE_EPI_BIAS_RESIDUAL_RMSNORM = 9
GE_EPI_BIAS_RESIDUAL_LAYERNORM = 10
GE_EPI_DW_DRELU_BGRAD = 11
# ge_dtype_t
GE_F16 = 0
GE_F32 = 1
GE_BF16 = 2
# ge_major_t
GE_K_MAJOR = 0
GE_MN_MAJOR = 1
# ge_dlayout_t
GE_D_ROW = 0
GE_D_COL = 1
# ge_plan_attr_t
GE_ATTR_STATIC_A = 0
# ge_path_t
GE_PATH_TC_GEMM = 0
GE_PATH_GEMV = 1
GE_PATH_DRELU = 2

EPILOGUE_BY_NAME = {"none": GE_EPI_NONE, "bias": GE_EPI_BIAS, "relu_bias": GE_EPI_RELU_BIAS,
                    "gelu_bias": GE_EPI_GELU_BIAS, "relu_aux_bias": GE_EPI_RELU_AUX_BIAS,
                    "drelu_bgrad": GE_EPI_DRELU_BGRAD, "gelu_erf_bias": GE_EPI_GELU_ERF_BIAS,
                    "gelu_aux_bias": GE_EPI_GELU_AUX_BIAS, "dgelu_bgrad": GE_EPI_DGELU_BGRAD,
                    "rmsnorm": GE_EPI_BIAS_RESIDUAL_RMSNORM, "layernorm": GE_EPI_BIAS_RESIDUAL_LAYERNORM,
                    "dw_drelu_bgrad": GE_EPI_DW_DRELU_BGRAD}

# Every function the header declares (checked against include/ge.h by a test).
ABI_FUNCTIONS = ("ge_plan_create", "ge_execute", "ge_execute_unfused", "ge_plan_free",
                 "ge_aux_bytes", "ge_aux_ld", "ge_plan_path", "ge_plan_tile_n",
                 "ge_get_last_device_error", "ge_status_string", "ge_debug_wait_timeout",
                 "ge_version", "ge_drelu_bgrad_static", "ge_plan_set_attr",
                 "ge_plan_autotune", "ge_plan_config", "ge_execute_norm", "ge_execute_norm_unfused",
                 "ge_autotune_cache_clear", "ge_execute_chain", "ge_debug_checks", "ge_debug_check_probe",
                 "ge_plan_stream_k_tiles")


class ge_layout_t(ctypes.Structure):
    _fields_ = [("a", ctypes.c_int), ("b", ctypes.c_int), ("d", ctypes.c_int),
                ("lda", ctypes.c_int64), ("ldb", ctypes.c_int64), ("ldd", ctypes.c_int64),
                ("ld_aux", ctypes.c_int64)]


class GeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {ge_status_string(status)}")


_lock = threading.Lock()
_lib = None


def load_library():
    """Load the CUDA library (raises if it is missing: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build() "
                               "(nvcc for sm_103a) first")
        lib = ctypes.CDLL(LIB_PATH)
        i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
        lib.ge_plan_create.argtypes = [ctypes.POINTER(vp), i64, i64, i64, i32, i32, i32, i32, i32,
                                       ctypes.POINTER(ge_layout_t)]
        lib.ge_plan_create.restype = i32
        lib.ge_execute.argtypes = [vp, vp, vp, vp, vp, vp, vp]
        lib.ge_execute.restype = i32
        lib.ge_execute_unfused.argtypes = [vp, vp, vp, vp, vp, vp, vp]
        lib.ge_execute_unfused.restype = i32
        lib.ge_autotune_cache_clear.argtypes = []
        lib.ge_autotune_cache_clear.restype = None
        for fn in (lib.ge_execute_norm, lib.ge_execute_norm_unfused):
            fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp]
            fn.restype = i32
        lib.ge_plan_free.argtypes = [vp]
        lib.ge_plan_free.restype = i32
        lib.ge_aux_bytes.argtypes = [vp]
        lib.ge_aux_bytes.restype = sz
        lib.ge_aux_ld.argtypes = [vp]
        lib.ge_aux_ld.restype = i64
        lib.ge_plan_path.argtypes = [vp]
        lib.ge_plan_path.restype = i32
        lib.ge_plan_tile_n.argtypes = [vp]
        lib.ge_plan_tile_n.restype = i32
        lib.ge_get_last_device_error.argtypes = [vp]
        lib.ge_get_last_device_error.restype = i32
        lib.ge_status_string.argtypes = [i32]
        lib.ge_status_string.restype = ctypes.c_char_p
        lib.ge_debug_wait_timeout.argtypes = [vp, i64, vp]
        lib.ge_debug_wait_timeout.restype = i32
        lib.ge_drelu_bgrad_static.argtypes = [i64, i64, i32, i64, i64, vp, vp, vp, vp, vp]
        lib.ge_drelu_bgrad_static.restype = i32
        lib.ge_plan_set_attr.argtypes = [vp, i32, i64]
        lib.ge_plan_set_attr.restype = i32
        lib.ge_plan_autotune.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32]
        lib.ge_plan_autotune.restype = i32
        lib.ge_plan_config.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i32)]
        lib.ge_plan_config.restype = i32
        lib.ge_plan_stream_k_tiles.argtypes = [vp]
        lib.ge_plan_stream_k_tiles.restype = i32
        lib.ge_execute_chain.argtypes = [vp, i64, ctypes.POINTER(vp), ctypes.POINTER(vp), vp, vp, vp]
        lib.ge_execute_chain.restype = i32
        lib.ge_debug_checks.argtypes = []
        lib.ge_debug_checks.restype = i32
        lib.ge_debug_check_probe.argtypes = [vp, vp]
        lib.ge_debug_check_probe.restype = i32
        lib.ge_version.argtypes = []
        lib.ge_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str):
    if status != GE_OK:
        raise GeError(status, where)


def ge_status_string(status: int) -> str:
    return load_library().ge_status_string(int(status)).decode()


def ge_version() -> str:
    return load_library().ge_version().decode()


def ge_plan_create(M: int, N: int, K: int, a: int = GE_F16, b: int = GE_F16, d: int = GE_F16,
                   compute: int = GE_F32, epi: int = GE_EPI_BIAS, layout: ge_layout_t | None = None,
                   *, raw: bool = False):
    """Returns the plan handle (an int); with raw=True returns (status, handle)."""
    lib = load_library()
    out = ctypes.c_void_p()
    st = lib.ge_plan_create(ctypes.byref(out), int(M), int(N), int(K), int(a), int(b), int(d),
                            int(compute), int(epi), ctypes.byref(layout) if layout is not None else None)
    if raw:
        return st, out.value
    _check(st, "ge_plan_create")
    return out.value


def ge_execute(plan, A, B, bias, D, aux=None, stream=None, *, raw: bool = False):
    st = load_library().ge_execute(plan, _ptr(A), _ptr(B), _ptr(bias), _ptr(D), _ptr(aux),
                                   _stream(stream))
    if raw:
        return st
    _check(st, "ge_execute")


def ge_autotune_cache_clear():
    load_library().ge_autotune_cache_clear()


def ge_execute_norm(plan, A, B, bias, residual, gamma, beta, H, Y, eps=1e-5, stream=None, *,
                    raw: bool = False, unfused: bool = False):
    """MatMul + bias + residual + RMSNorm/LayerNorm (``unfused=True``: the
    separate-kernel flow ge_execute_norm_unfused)."""
    lib = load_library()
    fn = lib.ge_execute_norm_unfused if unfused else lib.ge_execute_norm
    st = fn(plan, _ptr(A), _ptr(B), _ptr(bias), _ptr(residual), _ptr(gamma), _ptr(beta), _ptr(H), _ptr(Y),
            float(eps), _stream(stream))
    if raw:
        return st
    _check(st, "ge_execute_norm_unfused" if unfused else "ge_execute_norm")


def ge_execute_unfused(plan, A, B, bias, D, aux=None, stream=None, *, raw: bool = False):
    st = load_library().ge_execute_unfused(plan, _ptr(A), _ptr(B), _ptr(bias), _ptr(D), _ptr(aux),
                                           _stream(stream))
    if raw:
        return st
    _check(st, "ge_execute_unfused")


def ge_execute_chain(plan, As, biases, X, Y, stream=None, *, raw: bool = False):
    """A stack of len(As) decode projections in one launch (see include/ge.h);
    ``biases`` may be None for a NONE plan."""
    n = len(As)
    arr_a = (ctypes.c_void_p * max(n, 1))(*[_ptr(a) for a in As])
    arr_b = None
    if biases is not None:
        arr_b = (ctypes.c_void_p * max(n, 1))(*[_ptr(b) for b in biases])
    st = load_library().ge_execute_chain(plan, n, arr_a, arr_b, _ptr(X), _ptr(Y), _stream(stream))
    if raw:
        return st
    _check(st, "ge_execute_chain")


def ge_plan_set_attr(plan, attr: int, value: int, *, raw: bool = False):
    st = load_library().ge_plan_set_attr(plan, int(attr), int(value))
    if raw:
        return st
    _check(st, "ge_plan_set_attr")


def ge_plan_autotune(plan, A, B, bias, D, aux=None, stream=None, reps: int = 5, *, raw: bool = False):
    st = load_library().ge_plan_autotune(plan, _ptr(A), _ptr(B), _ptr(bias), _ptr(D), _ptr(aux),
                                         _stream(stream), int(reps))
    if raw:
        return st
    _check(st, "ge_plan_autotune")


def ge_plan_config(plan):
    """(path, block_n, pair, split) of the plan."""
    bn, pr, sp = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    path = load_library().ge_plan_config(plan, ctypes.byref(bn), ctypes.byref(pr), ctypes.byref(sp))
    return path, bn.value, pr.value, sp.value


def ge_plan_stream_k_tiles(plan) -> int:
    """Tiles the plan computes stream-K (0: none)."""
    return int(load_library().ge_plan_stream_k_tiles(plan))


def ge_plan_free(plan):
    _check(load_library().ge_plan_free(plan), "ge_plan_free")


def ge_aux_bytes(plan) -> int:
    return int(load_library().ge_aux_bytes(plan))


def ge_aux_ld(plan) -> int:
    return int(load_library().ge_aux_ld(plan))


def ge_plan_path(plan) -> int:
    return int(load_library().ge_plan_path(plan))


def ge_plan_tile_n(plan) -> int:
    return int(load_library().ge_plan_tile_n(plan))


def ge_get_last_device_error(plan) -> int:
    return int(load_library().ge_get_last_device_error(plan))


def ge_debug_wait_timeout(plan, budget_cycles: int, stream=None) -> int:
    return int(load_library().ge_debug_wait_timeout(plan, int(budget_cycles), _stream(stream)))


def ge_debug_checks() -> bool:
    return bool(load_library().ge_debug_checks())


def ge_debug_check_probe(plan, stream=None) -> int:
    return int(load_library().ge_debug_check_probe(plan, _stream(stream)))


def ge_drelu_bgrad_static(M: int, N: int, d: int, ldd: int, ld_aux: int, dY, aux, dZ, bgrad,
                          stream=None, *, raw: bool = False):
    """DRELU_BGRAD with no allocation (scratch in a fixed device array); see
    include/ge.h for the callers it serves and its size limit."""
    st = load_library().ge_drelu_bgrad_static(int(M), int(N), int(d), int(ldd), int(ld_aux), _ptr(dY),
                                              _ptr(aux), _ptr(dZ), _ptr(bgrad), _stream(stream))
    if raw:
        return st
    _check(st, "ge_drelu_bgrad_static")


def make_layout(a: int = GE_K_MAJOR, b: int = GE_MN_MAJOR, d: int = GE_D_ROW, lda: int = 0,
                ldb: int = 0, ldd: int = 0, ld_aux: int = 0) -> ge_layout_t:
    return ge_layout_t(a, b, d, lda, ldb, ldd, ld_aux)


class Plan:
    """Context-managed plan: ``with Plan(M, N, K, epi, layout) as p: p.execute(...)``.
    ``dtype`` is the element type of A, B, D and the bias (GE_F16 or GE_BF16)."""

    def __init__(self, M, N, K, epi=GE_EPI_BIAS, layout: ge_layout_t | None = None, dtype: int = GE_F16):
        self.M, self.N, self.K, self.epi, self.dtype = M, N, K, epi, dtype
        self.handle = ge_plan_create(M, N, K, dtype, dtype, dtype, epi=epi, layout=layout)

    def execute(self, A, B, bias, D, aux=None, stream=None):
        ge_execute(self.handle, A, B, bias, D, aux, stream)

    def set_attr(self, attr: int, value: int):
        ge_plan_set_attr(self.handle, attr, value)

    def autotune(self, A, B, bias, D, aux=None, stream=None, reps: int = 5):
        ge_plan_autotune(self.handle, A, B, bias, D, aux, stream, reps)

    @property
    def config(self):
        return ge_plan_config(self.handle)

    @property
    def stream_k_tiles(self) -> int:
        return ge_plan_stream_k_tiles(self.handle)

    def execute_chain(self, As, biases, X, Y, stream=None):
        ge_execute_chain(self.handle, As, biases, X, Y, stream)

    def execute_unfused(self, A, B, bias, D, aux=None, stream=None):
        ge_execute_unfused(self.handle, A, B, bias, D, aux, stream)

    def execute_norm(self, A, B, bias, residual, gamma, beta, H, Y, eps=1e-5, stream=None, unfused=False):
        ge_execute_norm(self.handle, A, B, bias, residual, gamma, beta, H, Y, eps, stream, unfused=unfused)

    @property
    def aux_bytes(self) -> int:
        return ge_aux_bytes(self.handle)

    @property
    def aux_ld(self) -> int:
        return ge_aux_ld(self.handle)

    @property
    def path(self) -> int:
        return ge_plan_path(self.handle)

    @property
    def tile_n(self) -> int:
        return ge_plan_tile_n(self.handle)

    def free(self):
        if self.handle:
            ge_plan_free(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.free()

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass
