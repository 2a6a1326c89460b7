"""GELU_AUX_BIAS (tanh-GELU forward that also keeps z = A.B + bias) and its
backward DGELU_BGRAD (dZ = dY * gelu'(z), fp32 bias gradient), on the GPU
against the oracle: every operand major and D layout, ragged edges, 2-SM
tiles with a split-K tail, fp16 and bf16, the unfused baseline, and the
standalone and GEMM-epilogue forms of the backward."""
import numpy as np
import pytest
import torch

import gemm_epilogues_gb300 as ge
from gemm_epilogues_gb300.inputs import TORCH_DTYPE, f16_tensor

from _util import GE_DT, bits, check_bgrad, check_f16

pytestmark = pytest.mark.gpu

MAJ = {"k": ge.GE_K_MAJOR, "m": ge.GE_MN_MAJOR, "n": ge.GE_MN_MAJOR}


def _pad8(x):
    return (x + 7) // 8 * 8


def run_forward(oracle, M, N, K, am, bm, dl, seed, dtype="f16", unfused=False, ld_zaux=0):
    t = TORCH_DTYPE[dtype]
    a_shape = (M, K) if am == "k" else (K, M)
    b_shape = (N, K) if bm == "k" else (K, N)
    rows, cols = (M, N) if dl == "row" else (N, M)
    lda, ldb, ldd = _pad8(a_shape[1]), _pad8(b_shape[1]), _pad8(cols)
    ldz = ld_zaux or _pad8(cols)
    A = f16_tensor((a_shape[0], lda), seed + 1, dtype=t).cuda()
    B = f16_tensor((b_shape[0], ldb), seed + 2, dtype=t).cuda()
    bias = f16_tensor((M,), seed + 3, dtype=t).cuda()
    A[:, a_shape[1]:] = float("nan")
    B[:, b_shape[1]:] = float("nan")
    L = ge.make_layout(MAJ[am], MAJ[bm], ge.GE_D_ROW if dl == "row" else ge.GE_D_COL, lda, ldb, ldd, ld_zaux)
    with ge.Plan(M, N, K, ge.GE_EPI_GELU_AUX_BIAS, L, dtype=GE_DT[dtype]) as p:
        assert p.path == ge.GE_PATH_TC_GEMM
        assert p.aux_ld == ldz and p.aux_bytes == rows * ldz * 2
        D = torch.full((rows, ldd), float("nan"), dtype=t, device="cuda")
        Z = torch.full((rows, ldz), float("nan"), dtype=t, device="cuda")
        (p.execute_unfused if unfused else p.execute)(A, B, bias, D, Z)
        torch.cuda.synchronize()
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
    ref = oracle.linear_forward(bits(A), bits(B), bits(bias), "gelu_aux_bias", M, N, K, a_major=am, b_major=bm,
                                d_layout=dl, lda=lda, ldb=ldb, ldd=ldd, ld_zaux=ldz, dtype=dtype)
    what = f"gelu_aux {M}x{N}x{K} {am}{bm}{dl} {dtype}{' unfused' if unfused else ''}"
    zref = ref["Z"].reshape(rows, ldd)[:, :cols]
    extra = None
    if unfused and dtype == "bf16":
        # the unfused flow rounds A.B to bf16 before the bias add
        b64 = oracle.f16_decode(bits(bias), dtype)
        extra = (2.0 ** -8 * np.abs(zref - (b64[:, None] if dl == "row" else b64[None, :]))).reshape(-1)
    got = bits(D).reshape(rows, ldd)[:, :cols].reshape(-1)
    check_f16(oracle, got, ref["D"].reshape(rows, ldd)[:, :cols].reshape(-1), what + " D", dtype, extra)
    gz = bits(Z).reshape(rows, ldz)[:, :cols].reshape(-1)
    check_f16(oracle, gz, ref["zaux"].reshape(rows, ldz)[:, :cols].reshape(-1), what + " z", dtype, extra)
    assert torch.isnan(D[:, cols:].float()).all() and torch.isnan(Z[:, cols:].float()).all(), \
        what + ": wrote past the logical columns"
    return Z


@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (129, 17, 72), (257, 1030, 1030)])
@pytest.mark.parametrize("am,bm,dl", [("k", "n", "row"), ("k", "k", "col"), ("m", "n", "row"), ("m", "k", "col")])
def test_gelu_aux_forward(oracle, M, N, K, am, bm, dl):
    run_forward(oracle, M, N, K, am, bm, dl, seed=300 + M)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_gelu_aux_pair_split_tail(oracle, monkeypatch, dtype):
    """2-SM tiles and a split-K tail (the fixup kernel writes z too)."""
    monkeypatch.setenv("GE_PAIR", "1")
    monkeypatch.setenv("GE_TILE_N", "256")
    run_forward(oracle, 1000, 2056, 520, "k", "n", "row", seed=310, dtype=dtype)
    run_forward(oracle, 513, 264, 4100, "k", "k", "col", seed=311, dtype=dtype)


def test_gelu_aux_decode_width_and_padded_ld(oracle):
    """N <= 16 stays on the tensor-core path (the GEMV has no aux output);
    a padded ld_aux leaves the padding untouched."""
    run_forward(oracle, 1000, 3, 1030, "k", "k", "col", seed=320, ld_zaux=1008)
    run_forward(oracle, 64, 16, 64, "k", "n", "row", seed=321, ld_zaux=24)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_gelu_aux_unfused(oracle, dtype):
    run_forward(oracle, 300, 520, 200, "k", "n", "row", seed=330, dtype=dtype, unfused=True)
    run_forward(oracle, 300, 517, 200, "k", "k", "col", seed=331, dtype=dtype, unfused=True)


def run_dgelu(oracle, M, N, K, dl, seed, dtype="f16", am="k", bm="k", inplace=False):
    """K == 0: standalone on a stored dY; K >= 1: applied to the product A.B."""
    t = TORCH_DTYPE[dtype]
    rows, cols = (M, N) if dl == "row" else (N, M)
    ldd, ldz = _pad8(cols), _pad8(cols + 3)
    # z: pre-activations of a typical spread (what GELU_AUX_BIAS stores)
    Z = f16_tensor((rows, ldz), seed + 5, "normal", 2.0, dtype=t).cuda()
    L = ge.make_layout(MAJ[am], MAJ[bm], ge.GE_D_ROW if dl == "row" else ge.GE_D_COL, 0, 0, ldd, ldz)
    bgrad = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
    if K == 0:
        dY = f16_tensor((rows, ldd), seed + 4, "normal", 1.0, dtype=t).cuda()
        dY_host = dY.cpu()
        dZ = dY if inplace else torch.full_like(dY, float("nan"))
        with ge.Plan(M, N, 0, ge.GE_EPI_DGELU_BGRAD, L, dtype=GE_DT[dtype]) as p:
            assert p.path == ge.GE_PATH_DRELU
            p.execute(dY, None, bgrad, dZ, Z)
            torch.cuda.synchronize()
            assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
        ref_dz, ref_bg = oracle.dgelu_bgrad(bits(dY_host), bits(Z), M, N, d_layout=dl, ldd=ldd, ld_zaux=ldz,
                                            dtype=dtype)
    else:
        a_shape = (M, K) if am == "k" else (K, M)
        b_shape = (N, K) if bm == "k" else (K, N)
        lda, ldb = _pad8(a_shape[1]), _pad8(b_shape[1])
        L = ge.make_layout(MAJ[am], MAJ[bm], ge.GE_D_ROW if dl == "row" else ge.GE_D_COL, lda, ldb, ldd, ldz)
        A = f16_tensor((a_shape[0], lda), seed + 1, "normal", K ** -0.5, dtype=t).cuda()
        B = f16_tensor((b_shape[0], ldb), seed + 2, dtype=t).cuda()
        dZ = torch.full((rows, ldd), float("nan"), dtype=t, device="cuda")
        with ge.Plan(M, N, K, ge.GE_EPI_DGELU_BGRAD, L, dtype=GE_DT[dtype]) as p:
            assert p.path == ge.GE_PATH_TC_GEMM
            p.execute(A, B, bgrad, dZ, Z)
            torch.cuda.synchronize()
            assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
        ref_dz, ref_bg = oracle.gemm_dgelu_bgrad(bits(A), bits(B), bits(Z), M, N, K, a_major=am, b_major=bm,
                                                 d_layout=dl, lda=lda, ldb=ldb, ldd=ldd, ld_zaux=ldz,
                                                 dtype=dtype)
    what = f"dgelu {M}x{N}x{K} {dl} {dtype}"
    got = bits(dZ).reshape(rows, ldd)[:, :cols].reshape(-1)
    check_f16(oracle, got, ref_dz.reshape(rows, ldd)[:, :cols].reshape(-1), what, dtype)
    if K == 0 and not inplace:
        assert torch.isnan(dZ[:, cols:].float()).all(), what + ": wrote past the logical columns"
    dzf = oracle.f16_decode(ref_dz, dtype).reshape(rows, ldd)[:, :cols]
    abs_sum = np.abs(dzf).sum(axis=0 if dl == "col" else 1)
    check_bgrad(bgrad.cpu().numpy(), ref_bg, abs_sum, what + " bgrad")
    return bgrad


@pytest.mark.parametrize("M,N", [(1, 1), (37, 5), (300, 1000), (2050, 129), (777, 4100)])
@pytest.mark.parametrize("dl", ["row", "col"])
def test_dgelu_standalone(oracle, M, N, dl):
    run_dgelu(oracle, M, N, 0, dl, seed=340 + M)


@pytest.mark.parametrize("dl", ["row", "col"])
def test_dgelu_standalone_bf16_and_inplace(oracle, dl):
    run_dgelu(oracle, 300, 1000, 0, dl, seed=350, dtype="bf16")
    run_dgelu(oracle, 513, 700, 0, dl, seed=351, inplace=True)


def test_dgelu_standalone_deterministic(oracle):
    b1 = run_dgelu(oracle, 1500, 4000, 0, "col", seed=355)
    b2 = run_dgelu(oracle, 1500, 4000, 0, "col", seed=355)
    assert torch.equal(b1, b2)


@pytest.mark.parametrize("M,N,K", [(1, 1, 8), (37, 45, 72), (300, 520, 200), (257, 129, 1030)])
@pytest.mark.parametrize("am,bm,dl", [("k", "n", "row"), ("k", "k", "col"), ("m", "n", "row"), ("m", "k", "col")])
def test_gemm_dgelu_bgrad(oracle, M, N, K, am, bm, dl):
    run_dgelu(oracle, M, N, K, dl, seed=360 + K, am=am, bm=bm)


@pytest.mark.parametrize("dl", ["row", "col"])
def test_gemm_dgelu_bgrad_pair_and_bf16(oracle, monkeypatch, dl):
    monkeypatch.setenv("GE_PAIR", "1")
    monkeypatch.setenv("GE_TILE_N", "256")
    run_dgelu(oracle, 700, 900, 328, dl, seed=370, bm="k" if dl == "col" else "n")
    run_dgelu(oracle, 700, 900, 328, dl, seed=371, dtype="bf16", bm="k" if dl == "col" else "n")
