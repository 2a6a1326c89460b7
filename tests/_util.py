"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and compute the oracle's answer (whole problem or sampled stored rows)."""
from __future__ import annotations

import numpy as np
import torch

import gemm_epilogues_gb300 as ge
from gemm_epilogues_gb300.inputs import TORCH_DTYPE, Workload

MAJOR = {"k": ge.GE_K_MAJOR, "m": ge.GE_MN_MAJOR, "n": ge.GE_MN_MAJOR}
DLAY = {"row": ge.GE_D_ROW, "col": ge.GE_D_COL}
GE_DT = {"f16": ge.GE_F16, "bf16": ge.GE_BF16}

# Tolerances (16-bit outputs: |err| <= 1e-2 * max(1, |ref|); mask bit-exact
# where |pre-activation| > 1e-3; fp32 bias gradient: relative 1e-4). For bf16
# the same bound holds: one bf16 step is at most 2^-7 = 0.0078 of the value.
F16_REL = 1e-2
MASK_BAND = 1e-3
BGRAD_REL = 1e-4


def bits(t: torch.Tensor) -> np.ndarray:
    """fp16/bf16 tensor (any device) -> numpy uint16 bit patterns (flat)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1)


def layout_of(w: Workload, lda=0, ldb=0, ldd=0, ld_aux=0):
    return ge.make_layout(MAJOR[w.a_major], MAJOR[w.b_major], DLAY[w.d_layout], lda, ldb, ldd, ld_aux)


def gpu_forward(w: Workload, A, B, bias, *, unfused=False, ld=None, stream=None):
    """Run D = act(A.B + bias) on the GPU through the C ABI. A, B, bias are
    CUDA fp16 tensors in storage layout. Returns (D, aux, plan path)."""
    ld = ld or {}
    L = layout_of(w, ld.get("lda", 0), ld.get("ldb", 0), ld.get("ldd", 0))
    with ge.Plan(w.M, w.N, w.K, ge.EPILOGUE_BY_NAME[w.epilogue], L, dtype=GE_DT[w.dtype]) as p:
        rows, cols = w.d_shape()
        ldd = ld.get("ldd", 0) or cols
        D = torch.full((rows, ldd), float("nan"), dtype=TORCH_DTYPE[w.dtype], device=A.device)
        aux = None
        if w.epilogue == "relu_aux_bias":
            aux = torch.full((p.aux_bytes // 4,), 0xA5A5A5A5 - 2**32, dtype=torch.int32, device=A.device)
        bias_arg = bias if w.epilogue != "none" else None
        if unfused:
            p.execute_unfused(A, B, bias_arg, D, aux, stream)
        else:
            p.execute(A, B, bias_arg, D, aux, stream)
        torch.cuda.synchronize()
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
        return D, aux, p.path, p.aux_ld


def oracle_full(oracle, w: Workload, A, B, bias, ld=None):
    ld = ld or {}
    return oracle.linear_forward(bits(A), bits(B), bits(bias) if w.epilogue != "none" else None,
                                 w.epilogue, w.M, w.N, w.K, a_major=w.a_major, b_major=w.b_major,
                                 d_layout=w.d_layout, lda=ld.get("lda"), ldb=ld.get("ldb"),
                                 ldd=ld.get("ldd"), dtype=w.dtype)


def oracle_rows(oracle, w: Workload, A, B, bias, rows: np.ndarray):
    """Oracle on the sub-problem made of the given stored rows of D: for a
    row-major D the rows are m (A's rows and bias entries), for a
    column-major D they are n (B's columns). Returns the oracle dict; its
    stored rows follow `rows`."""
    idx = torch.as_tensor(rows, dtype=torch.long, device=A.device)
    if w.d_layout == "row":
        A_sub = A.index_select(0 if w.a_major == "k" else 1, idx)
        sub = dict(M=len(rows), N=w.N, A=A_sub, B=B, bias=bias.index_select(0, idx))
    else:
        B_sub = B.index_select(0 if w.b_major == "k" else 1, idx)
        sub = dict(M=w.M, N=len(rows), A=A, B=B_sub, bias=bias)
    return oracle.linear_forward(bits(sub["A"]), bits(sub["B"]),
                                 bits(sub["bias"]) if w.epilogue != "none" else None, w.epilogue,
                                 sub["M"], sub["N"], w.K, a_major=w.a_major, b_major=w.b_major,
                                 d_layout=w.d_layout, dtype=w.dtype)


def check_f16(oracle, got_bits: np.ndarray, ref_bits: np.ndarray, what: str, dtype: str = "f16",
              extra_tol=None):
    """16-bit output within F16_REL * max(1, |ref|), plus `extra_tol` (per
    element) where a path rounds an intermediate to 16 bits."""
    got = oracle.f16_decode(got_bits, dtype)
    ref = oracle.f16_decode(ref_bits, dtype)
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    tol = F16_REL * np.maximum(1.0, np.abs(ref))
    if extra_tol is not None:
        tol = tol + extra_tol
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance, worst err "
                           f"{err.max():.4g} at {int(err.argmax())} (ref {ref[err.argmax()]:.6g})")
    return float(err.max())


def mask_bits(words: np.ndarray, rows: int, ld_aux: int, cols: int) -> np.ndarray:
    w = words.reshape(rows, ld_aux)[:, : (cols + 31) // 32]
    b = np.unpackbits(w.view(np.uint8).reshape(rows, -1), axis=1, bitorder="little")
    return b[:, :cols]


def check_mask(got_words, ref_words, Z, rows, cols, ld_aux, what, band=None):
    """Mask bits equal wherever |z| is outside the band (MASK_BAND, or a
    per-element `band` [rows, cols] for a path that rounds z first)."""
    g = mask_bits(got_words, rows, ld_aux, cols)
    r = mask_bits(ref_words, rows, ld_aux, cols)
    z = Z.reshape(rows, -1)[:, :cols]
    sure = np.abs(z) > (MASK_BAND if band is None else band)
    assert np.array_equal(g[sure], r[sure]), f"{what}: mask differs outside the |z| <= 1e-3 band"
    # bits past the end of each row (up to the 128-column padding) are zero
    gw = got_words.reshape(rows, ld_aux)
    pad_words = (cols + 127) // 128 * 4
    full = np.unpackbits(gw[:, :pad_words].view(np.uint8).reshape(rows, -1), axis=1, bitorder="little")
    assert not full[:, cols:].any(), f"{what}: padding bits set"


def check_bgrad(got: np.ndarray, ref: np.ndarray, abs_sum: np.ndarray, what: str):
    """fp32 bias gradient vs the fp64 oracle: per element
    |g - ref| <= 1e-4 * max(|ref|, sum|dZ| * 2^-7) (the second term keeps a
    sum that cancels to ~0 well-conditioned), and norm-wise
    max|g - ref| <= 1e-4 * max|ref|."""
    err = np.abs(got.astype(np.float64) - ref)
    tol = BGRAD_REL * np.maximum(np.abs(ref), abs_sum * 2.0 ** -7)
    bad = err > tol
    assert not bad.any(), f"{what}: {bad.sum()} bias-gradient entries outside tolerance (worst {err.max():.3g})"
    assert err.max() <= BGRAD_REL * max(np.abs(ref).max(), 1e-30), f"{what}: norm-wise error"
