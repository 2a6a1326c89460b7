"""MatMul + bias + residual + RMSNorm / LayerNorm on the GPU against the
oracle: H (the rounded residual stream) and Y, on the tensor-core and GEMV
paths, feature counts that span the register cache and a ragged tail, fp16
and bf16, H written over the residual and Y over H, and the unfused flow."""
import numpy as np
import pytest
import torch

import gemm_epilogues_gb300 as ge
from gemm_epilogues_gb300.inputs import TORCH_DTYPE, f16_tensor

from _util import GE_DT, bits, check_f16

pytestmark = pytest.mark.gpu

MAJ = {"k": ge.GE_K_MAJOR, "m": ge.GE_MN_MAJOR, "n": ge.GE_MN_MAJOR}
EPI = {"rmsnorm": ge.GE_EPI_BIAS_RESIDUAL_RMSNORM, "layernorm": ge.GE_EPI_BIAS_RESIDUAL_LAYERNORM}


def _pad8(x):
    return (x + 7) // 8 * 8


def run_norm(oracle, M, N, K, norm, seed, am="k", bm="k", dtype="f16", inplace=False, unfused=False, eps=1e-5):
    t = TORCH_DTYPE[dtype]
    a_shape = (M, K) if am == "k" else (K, M)
    b_shape = (N, K) if bm == "k" else (K, N)
    lda, ldb, ldd = _pad8(a_shape[1]), _pad8(b_shape[1]), _pad8(M)
    A = f16_tensor((a_shape[0], lda), seed + 1, "normal", K ** -0.5, dtype=t).cuda()
    B = f16_tensor((b_shape[0], ldb), seed + 2, dtype=t).cuda()
    bias = f16_tensor((M,), seed + 3, "normal", 0.3, dtype=t).cuda()
    res = f16_tensor((N, ldd), seed + 4, dtype=t).cuda()
    gamma = (1 + f16_tensor((M,), seed + 5, "normal", 0.2, dtype=torch.float32)).to(t).cuda()
    beta = f16_tensor((M,), seed + 6, "normal", 0.2, dtype=t).cuda()
    res_host = res.cpu()
    L = ge.make_layout(MAJ[am], MAJ[bm], ge.GE_D_COL, lda, ldb, ldd)
    with ge.Plan(M, N, K, EPI[norm], L, dtype=GE_DT[dtype]) as p:
        assert p.path == (ge.GE_PATH_GEMV if N <= 16 and am == "k" and bm == "k" else ge.GE_PATH_TC_GEMM)
        bt = beta if norm == "layernorm" else None
        if inplace:
            # H written over the residual buffer ...
            H = res
            Y = torch.full((N, ldd), float("nan"), dtype=t, device="cuda")
            p.execute_norm(A, B, bias, res, gamma, bt, H, Y, eps)
            # ... and, in a second call on the same inputs, Y written over H
            res2 = res_host.cuda()
            HY = torch.full((N, ldd), float("nan"), dtype=t, device="cuda")
            p.execute_norm(A, B, bias, res2, gamma, bt, HY, HY, eps)
            torch.cuda.synchronize()
            assert torch.equal(HY.view(torch.int16), Y.view(torch.int16)), "Y over H differs"
        else:
            H = torch.full((N, ldd), float("nan"), dtype=t, device="cuda")
            Y = torch.full((N, ldd), float("nan"), dtype=t, device="cuda")
            p.execute_norm(A, B, bias, res, gamma, bt, H, Y, eps, unfused=unfused)
        torch.cuda.synchronize()
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
    refH, refY = oracle.linear_norm(bits(A), bits(B), bits(bias), bits(res_host), bits(gamma), bits(beta), norm,
                                    M, N, K, eps=eps, a_major=am, b_major=bm, d_layout="col", lda=lda, ldb=ldb,
                                    ldd=ldd, dtype=dtype)
    what = f"{norm} {M}x{N}x{K} {am}{bm} {dtype}{' unfused' if unfused else ''}{' inplace' if inplace else ''}"
    extra = None
    if unfused and dtype == "bf16":
        # the unfused flow rounds A.B and A.B + bias to bf16 before the residual add
        h = oracle.f16_decode(refH, dtype).reshape(N, ldd)[:, :M]
        extra = (2.0 ** -7 * (np.abs(h) + 4)).reshape(-1)
    sl = lambda x: x.reshape(N, ldd)[:, :M].reshape(-1)
    check_f16(oracle, sl(bits(H)), sl(refH), what + " H", dtype, extra)
    # Y is normalised from the stored (rounded) H: that rounding, relative
    # 2^-11 (fp16) or 2^-8 (bf16) of |h|, passes through rstd * gamma.
    check_f16(oracle, sl(bits(Y)), sl(refY), what + " Y", dtype, extra)
    if not inplace:
        assert torch.isnan(H[:, M:].float()).all() and torch.isnan(Y[:, M:].float()).all(), \
            what + ": wrote past the features"


@pytest.mark.parametrize("norm", ["rmsnorm", "layernorm"])
@pytest.mark.parametrize("M,N,K", [(4096, 300, 512), (1000, 129, 200), (1003, 77, 96), (4100, 64, 64),
                                   (9000, 40, 64)])
def test_norm_tensor_core(oracle, norm, M, N, K):
    run_norm(oracle, M, N, K, norm, seed=400 + M + N)


@pytest.mark.parametrize("norm", ["rmsnorm", "layernorm"])
@pytest.mark.parametrize("N", [1, 3, 16])
def test_norm_decode_gemv(oracle, norm, N):
    run_norm(oracle, 4096, N, 4096, norm, seed=410 + N)


@pytest.mark.parametrize("norm", ["rmsnorm", "layernorm"])
def test_norm_layouts_bf16_inplace(oracle, norm):
    run_norm(oracle, 2048, 300, 256, norm, seed=420, am="m", bm="n")
    run_norm(oracle, 2048, 300, 256, norm, seed=421, dtype="bf16")
    run_norm(oracle, 2048, 300, 256, norm, seed=422, inplace=True)
    run_norm(oracle, 4096, 1, 4096, norm, seed=423, dtype="bf16", inplace=True)


@pytest.mark.parametrize("norm", ["rmsnorm", "layernorm"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_norm_unfused(oracle, norm, dtype):
    run_norm(oracle, 2048, 300, 256, norm, seed=430, dtype=dtype, unfused=True)
    run_norm(oracle, 1003, 77, 96, norm, seed=431, dtype=dtype, unfused=True)  # ragged rows of H


def test_norm_pair_tiles_split_tail(oracle, monkeypatch):
    monkeypatch.setenv("GE_PAIR", "1")
    monkeypatch.setenv("GE_TILE_N", "256")
    run_norm(oracle, 2056, 1000, 520, "layernorm", seed=440)


def test_norm_rejects_bad_calls():
    L = ge.make_layout(ge.GE_K_MAJOR, ge.GE_K_MAJOR, ge.GE_D_COL)
    with ge.Plan(256, 64, 64, ge.GE_EPI_BIAS_RESIDUAL_LAYERNORM, L) as p:
        A = torch.ones(256, 64, dtype=torch.float16, device="cuda")
        B = torch.ones(64, 64, dtype=torch.float16, device="cuda")
        v = torch.ones(256, dtype=torch.float16, device="cuda")
        H = torch.empty(64, 256, dtype=torch.float16, device="cuda")
        assert ge.ge_execute(p.handle, A, B, v, H, None, raw=True) == ge.GE_ERR_UNSUPPORTED
        assert ge.ge_execute_norm(p.handle, A, B, v, H, v, None, H, H, raw=True) == ge.GE_ERR_INVALID_ARG
        assert ge.ge_execute_norm(p.handle, A, B, v, H, v, v, H, H, eps=-1.0, raw=True) == ge.GE_ERR_INVALID_ARG
        assert ge.ge_execute_norm(p.handle, A, B, v, H, v, v, H, H, raw=True, unfused=True) == \
            ge.GE_ERR_INVALID_ARG  # H over the residual needs the fused path
        assert ge.ge_execute_norm(p.handle, A, B, v, H, v, v, H, H, raw=True) == ge.GE_OK
        torch.cuda.synchronize()


def _norm_given(oracle, A, B, bias, res, gamma, beta, norm, M, N, K, what, unfused=False):
    """Run the norm fusion on given fp16 inputs (A [M,K], B [N,K] K-major,
    residual [N,M]) and compare H and Y with the oracle."""
    L = ge.make_layout(ge.GE_K_MAJOR, ge.GE_K_MAJOR, ge.GE_D_COL)
    with ge.Plan(M, N, K, EPI[norm], L) as p:
        H = torch.full((N, M), float("nan"), dtype=torch.float16, device="cuda")
        Y = torch.full((N, M), float("nan"), dtype=torch.float16, device="cuda")
        p.execute_norm(A, B, bias, res, gamma, beta if norm == "layernorm" else None, H, Y, 1e-5, unfused=unfused)
        torch.cuda.synchronize()
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
    refH, refY = oracle.linear_norm(bits(A), bits(B), bits(bias), bits(res), bits(gamma), bits(beta), norm, M, N, K,
                                    eps=1e-5, d_layout="col")
    check_f16(oracle, bits(H), refH, what + " H")
    check_f16(oracle, bits(Y), refY, what + " Y")
    return Y


@pytest.mark.parametrize("norm", ["rmsnorm", "layernorm"])
@pytest.mark.parametrize("N", [1, 5, 200])
def test_norm_constant_tokens(oracle, norm, N):
    """A = 0 and bias = 0, so h is the residual; each token's residual row is
    one constant (one token all zeros). LayerNorm then gives beta (zero
    deviation, rstd = 1/sqrt(eps) multiplies only rounding noise); RMSNorm
    gives c/sqrt(c^2 + eps) times gamma."""
    M, K = 1000, 64
    A = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    B = f16_tensor((N, K), 450, device="cuda")
    bias = torch.zeros(M, dtype=torch.float16, device="cuda")
    c = f16_tensor((N, 1), 451, "normal", 3.0, "cuda")
    c[0] = 0.0
    res = c.expand(N, M).contiguous()
    gamma = (1 + f16_tensor((M,), 452, "normal", 0.2, dtype=torch.float32)).half().cuda()
    beta = f16_tensor((M,), 453, "normal", 0.2, "cuda")
    for unfused in (False, True):
        _norm_given(oracle, A, B, bias, res, gamma, beta, norm, M, N, K,
                    f"{norm} constant tokens N={N}{' unfused' if unfused else ''}", unfused)


@pytest.mark.parametrize("norm", ["rmsnorm", "layernorm"])
@pytest.mark.parametrize("N", [3, 300])
def test_norm_large_offset(oracle, norm, N):
    """Residual rows around 1000 with a spread of a few units (A = 0 and bias
    = 0, values on the fp16 grid there, so h is stored without rounding): the
    mean is ~300 times the deviation, where a sum of squares less a squared
    mean in fp32 would put an error of a few percent into the variance."""
    M, K = 4096, 64
    A = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    B = f16_tensor((N, K), 461, device="cuda")
    bias = torch.zeros(M, dtype=torch.float16, device="cuda")
    x = f16_tensor((N, M), 463, "normal", 3.0, dtype=torch.float32).clamp_(-20, 20)
    res = (1000.0 + torch.round(2 * x) / 2).half().cuda()
    gamma = (1 + f16_tensor((M,), 464, "normal", 0.2, dtype=torch.float32)).half().cuda()
    beta = f16_tensor((M,), 465, "normal", 0.2, "cuda")
    for unfused in (False, True):
        _norm_given(oracle, A, B, bias, res, gamma, beta, norm, M, N, K,
                    f"{norm} offset 1000 N={N}{' unfused' if unfused else ''}", unfused)
