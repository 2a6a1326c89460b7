"""The later rows at the sizes the benchmark times, in its launch
configuration: the GELU_AUX_BIAS forward and the backward GEMM with the
DGELU_BGRAD epilogue at 11008 x 8192 x 4096, the standalone DGELU_BGRAD and
row-layout DRELU_BGRAD passes on 8192 x 11008, MatMul + bias + residual +
RMSNorm / LayerNorm at 4096 x 8192 x 4096, and the bf16 forward and dW GEMMs
of the MLP layer.

Where the oracle cannot run the whole product in seconds, it runs the
sub-problem that yields exactly the sampled outputs: a token's outputs depend
only on its own input row (and residual row), and a feature's bias gradient
only on its own weight row and its own column of z; the elementwise passes
are checked whole."""
import numpy as np
import pytest
import torch

import gemm_epilogues_gb300 as ge
from gemm_epilogues_gb300.inputs import f16_tensor, sample_rows

from _util import bits, check_bgrad, check_f16, check_mask

pytestmark = pytest.mark.gpu

M_MLP, T_TOK, D_IN = 11008, 8192, 4096
KK_COL = ge.make_layout(ge.GE_K_MAJOR, ge.GE_K_MAJOR, ge.GE_D_COL)


def _ok(p):
    torch.cuda.synchronize()
    assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK


def test_gelu_aux_forward_fullsize(oracle):
    M, N, K = M_MLP, T_TOK, D_IN
    A = f16_tensor((M, K), 5101, "normal", 1 / 64, "cuda")
    B = f16_tensor((N, K), 5102, "normal", 1.0, "cuda")
    bias = f16_tensor((M,), 5103, "normal", 0.141, "cuda")
    with ge.Plan(M, N, K, ge.GE_EPI_GELU_AUX_BIAS, KK_COL) as p:
        assert p.path == ge.GE_PATH_TC_GEMM
        ldz = p.aux_ld
        D = torch.empty((N, M), dtype=torch.float16, device="cuda")
        Z = torch.empty((N, ldz), dtype=torch.float16, device="cuda")
        p.execute(A, B, bias, D, Z)
        _ok(p)
    assert torch.isfinite(D.float()).all() and torch.isfinite(Z[:, :M].float()).all()
    rows = sample_rows(N)
    idx = torch.as_tensor(rows, device="cuda")
    ref = oracle.linear_forward(bits(A), bits(B.index_select(0, idx)), bits(bias), "gelu_aux_bias", M, len(rows),
                                K, a_major="k", b_major="k", d_layout="col", ld_zaux=ldz)
    check_f16(oracle, bits(D.index_select(0, idx)), ref["D"], "gelu_aux 11008x8192x4096 D")
    gz = bits(Z.index_select(0, idx)).reshape(len(rows), ldz)[:, :M].reshape(-1)
    check_f16(oracle, gz, ref["zaux"].reshape(len(rows), ldz)[:, :M].reshape(-1), "gelu_aux 11008x8192x4096 z")


def test_dgelu_backward_gemm_fullsize(oracle):
    """dZ = (W2 . G^T) * gelu'(z) with bgrad over all 8192 tokens: sampled
    tokens for dZ, sampled features for dZ's columns and the bias gradient."""
    M, N, K = M_MLP, T_TOK, D_IN
    W2 = f16_tensor((M, K), 5201, "normal", 1 / 64, "cuda")
    G = f16_tensor((N, K), 5202, "normal", 1.0, "cuda")
    Zs = f16_tensor((N, M), 5203, "normal", 2.0, "cuda")
    with ge.Plan(M, N, K, ge.GE_EPI_DGELU_BGRAD, KK_COL) as p:
        assert p.path == ge.GE_PATH_TC_GEMM
        dZ = torch.empty((N, M), dtype=torch.float16, device="cuda")
        bgrad = torch.empty(M, dtype=torch.float32, device="cuda")
        p.execute(W2, G, bgrad, dZ, Zs)
        _ok(p)
    assert torch.isfinite(dZ.float()).all() and torch.isfinite(bgrad).all()
    # tokens
    rows = sample_rows(N)
    ri = torch.as_tensor(rows, device="cuda")
    ref_dz, _ = oracle.gemm_dgelu_bgrad(bits(W2), bits(G.index_select(0, ri)), bits(Zs.index_select(0, ri)), M,
                                        len(rows), K, d_layout="col")
    check_f16(oracle, bits(dZ.index_select(0, ri)), ref_dz, "dgelu GEMM 11008x8192x4096 dZ (tokens)")
    # features: every token's contribution to the sampled bias-gradient entries
    feats = sample_rows(M, 64, seed=0x5EED)
    fi = torch.as_tensor(feats, device="cuda")
    zsub = Zs.index_select(1, fi).contiguous()
    ref_dz_f, ref_bg = oracle.gemm_dgelu_bgrad(bits(W2.index_select(0, fi)), bits(G), bits(zsub), len(feats), N, K,
                                               d_layout="col", ld_zaux=len(feats))
    check_f16(oracle, bits(dZ.index_select(1, fi).contiguous()), ref_dz_f, "dgelu GEMM dZ (features)")
    abs_sum = np.abs(oracle.f16_decode(ref_dz_f).reshape(N, len(feats))).sum(axis=0)
    check_bgrad(bgrad.index_select(0, fi).cpu().numpy(), ref_bg, abs_sum, "dgelu GEMM bgrad (features)")


def test_dgelu_standalone_fullsize(oracle):
    M, N = M_MLP, T_TOK
    dY = f16_tensor((N, M), 5301, "normal", 1.0, "cuda")
    Zs = f16_tensor((N, M), 5302, "normal", 2.0, "cuda")
    with ge.Plan(M, N, 0, ge.GE_EPI_DGELU_BGRAD, ge.make_layout(d=ge.GE_D_COL)) as p:
        dZ = torch.empty_like(dY)
        bgrad = torch.empty(M, dtype=torch.float32, device="cuda")
        p.execute(dY, None, bgrad, dZ, Zs)
        _ok(p)
    ref_dz, ref_bg = oracle.dgelu_bgrad(bits(dY), bits(Zs), M, N, d_layout="col")
    check_f16(oracle, bits(dZ), ref_dz, "dgelu dY[8192,11008] dZ")
    abs_sum = np.abs(oracle.f16_decode(ref_dz).reshape(N, M)).sum(axis=0)
    check_bgrad(bgrad.cpu().numpy(), ref_bg, abs_sum, "dgelu dY[8192,11008] bgrad")


def test_drelu_rows_fullsize(oracle):
    """Row-major D: dY[11008 features][8192 tokens], random mask words."""
    M, N = M_MLP, T_TOK
    ld_aux = (N + 127) // 128 * 4
    dY = f16_tensor((M, N), 5401, "normal", 1.0, "cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5402)
    aux = torch.randint(-2**31, 2**31 - 1, (M * ld_aux,), generator=gen, device="cuda", dtype=torch.int32)
    with ge.Plan(M, N, 0, ge.GE_EPI_DRELU_BGRAD, ge.make_layout(d=ge.GE_D_ROW)) as p:
        dZ = torch.empty_like(dY)
        bgrad = torch.empty(M, dtype=torch.float32, device="cuda")
        p.execute(dY, None, bgrad, dZ, aux)
        _ok(p)
    ref_dz, ref_bg = oracle.drelu_bgrad(bits(dY), aux.cpu().numpy().view(np.uint32), M, N, d_layout="row",
                                        ld_aux=ld_aux)
    assert np.array_equal(bits(dZ), ref_dz), "drelu rows dZ differs"
    abs_sum = np.abs(oracle.f16_decode(ref_dz).reshape(M, N)).sum(axis=1)
    check_bgrad(bgrad.cpu().numpy(), ref_bg, abs_sum, "drelu rows bgrad")


@pytest.mark.parametrize("norm", ["rmsnorm", "layernorm"])
def test_norm_fullsize(oracle, norm):
    M, N, K = 4096, 8192, 4096
    epi = ge.GE_EPI_BIAS_RESIDUAL_RMSNORM if norm == "rmsnorm" else ge.GE_EPI_BIAS_RESIDUAL_LAYERNORM
    A = f16_tensor((M, K), 5501, "normal", K ** -0.5, "cuda")
    X = f16_tensor((N, K), 5502, "normal", 1.0, "cuda")
    bias = f16_tensor((M,), 5503, "normal", 0.3, "cuda")
    res = f16_tensor((N, M), 5504, "normal", 1.0, "cuda")
    gamma = (1 + f16_tensor((M,), 5505, "normal", 0.2, dtype=torch.float32)).half().cuda()
    beta = f16_tensor((M,), 5506, "normal", 0.2, "cuda")
    bt = beta if norm == "layernorm" else None
    with ge.Plan(M, N, K, epi, KK_COL) as p:
        assert p.path == ge.GE_PATH_TC_GEMM
        H = torch.empty((N, M), dtype=torch.float16, device="cuda")
        Y = torch.empty((N, M), dtype=torch.float16, device="cuda")
        p.execute_norm(A, X, bias, res, gamma, bt, H, Y, 1e-5)
        _ok(p)
    assert torch.isfinite(Y.float()).all()
    rows = sample_rows(N)
    ri = torch.as_tensor(rows, device="cuda")
    refH, refY = oracle.linear_norm(bits(A), bits(X.index_select(0, ri)), bits(bias), bits(res.index_select(0, ri)),
                                    bits(gamma), bits(beta), norm, M, len(rows), K, eps=1e-5, d_layout="col")
    check_f16(oracle, bits(H.index_select(0, ri)), refH, f"{norm} 4096x8192x4096 H")
    check_f16(oracle, bits(Y.index_select(0, ri)), refY, f"{norm} 4096x8192x4096 Y")


def test_bf16_mlp_fullsize(oracle):
    """bf16 forward RELU_AUX_BIAS and dW at the MLP size (sampled)."""
    M, N, K = M_MLP, T_TOK, D_IN
    bf = torch.bfloat16
    A = f16_tensor((M, K), 5601, "normal", 1 / 64, "cuda", dtype=bf)
    X = f16_tensor((N, K), 5602, "normal", 1.0, "cuda", dtype=bf)
    bias = f16_tensor((M,), 5603, "normal", 0.141, "cuda", dtype=bf)
    with ge.Plan(M, N, K, ge.GE_EPI_RELU_AUX_BIAS, KK_COL, dtype=ge.GE_BF16) as p:
        ld_aux = p.aux_ld
        D = torch.empty((N, M), dtype=bf, device="cuda")
        aux = torch.empty(p.aux_bytes // 4, dtype=torch.int32, device="cuda")
        p.execute(A, X, bias, D, aux)
        _ok(p)
    assert torch.isfinite(D.float()).all() and (D >= 0).all()
    rows = sample_rows(N)
    ri = torch.as_tensor(rows, device="cuda")
    ref = oracle.linear_forward(bits(A), bits(X.index_select(0, ri)), bits(bias), "relu_aux_bias", M, len(rows), K,
                                a_major="k", b_major="k", d_layout="col", ld_aux=ld_aux, dtype="bf16")
    check_f16(oracle, bits(D.index_select(0, ri)), ref["D"], "bf16 fwd 11008x8192x4096", "bf16")
    gw = aux.view(N, ld_aux).index_select(0, ri).cpu().numpy().view(np.uint32).reshape(-1)
    check_mask(gw, ref["aux"], ref["Z"], len(rows), M, ld_aux, "bf16 fwd mask")
    # dW[11008, 4096] = dZ^T X: A = dZ read M-major, B = X read N-major, D row-major
    dZ = f16_tensor((N, M), 5604, "normal", 1.0, "cuda", dtype=bf)
    L = ge.make_layout(ge.GE_MN_MAJOR, ge.GE_MN_MAJOR, ge.GE_D_ROW)
    with ge.Plan(M, D_IN, N, ge.GE_EPI_NONE, L, dtype=ge.GE_BF16) as p:
        dW = torch.empty((M, D_IN), dtype=bf, device="cuda")
        p.execute(dZ, X, None, dW, None)
        _ok(p)
    mrows = sample_rows(M)
    mi = torch.as_tensor(mrows, device="cuda")
    ref = oracle.linear_forward(bits(dZ.index_select(1, mi).contiguous()), bits(X), None, "none", len(mrows), D_IN, N,
                                a_major="m", b_major="n", d_layout="row", dtype="bf16")
    check_f16(oracle, bits(dW.index_select(0, mi)), ref["D"], "bf16 dW 11008x4096x8192", "bf16")
