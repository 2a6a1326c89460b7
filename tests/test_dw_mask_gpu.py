"""DW_DRELU_BGRAD: the weight-gradient GEMM of a RELU_AUX_BIAS layer with the
ReLU backward applied to its A operand (dY), and the bias gradient. Every
test runs in both forms of the plan: the default two launches (the
standalone DRELU_BGRAD pass into the plan's dZ buffer, then the NONE GEMM on
it) and, with GE_DW_MASK=gemm, the mask applied inside the GEMM as the
kernel loads its operand (bias gradient reduced in the same pass). Against
the oracle (the pinned DRELU_BGRAD and GEMM steps composed): ragged extents
and pitches, 1-CTA and 2-SM tiles, split-K pieces, bf16, no bias-gradient
output; at the MLP size on sampled features, and bit-identical to the
unfused flow run by hand."""
import numpy as np
import pytest
import torch

import gemm_epilogues_gb300 as ge
from gemm_epilogues_gb300.inputs import TORCH_DTYPE, f16_tensor, sample_rows

from _util import GE_DT, bits, check_bgrad, check_f16

pytestmark = pytest.mark.gpu

MN, ROW = ge.GE_MN_MAJOR, ge.GE_D_ROW


@pytest.fixture(autouse=True, params=["two_launches", "in_gemm"])
def dw_mask_form(request, monkeypatch):
    if request.param == "in_gemm":
        monkeypatch.setenv("GE_DW_MASK", "gemm")
    else:
        monkeypatch.delenv("GE_DW_MASK", raising=False)
    return request.param


def _pad8(x):
    return (x + 7) // 8 * 8


def _inputs(M, N, K, seed, dtype, lda, ldx, ld_aux):
    t = TORCH_DTYPE[dtype]
    dY = f16_tensor((K, lda), seed + 1, dtype=t).cuda()
    X = f16_tensor((K, ldx), seed + 2, dtype=t).cuda()
    dY[:, M:] = float("nan")  # padding must never be read
    X[:, N:] = float("nan")
    g = torch.Generator(device="cuda")
    g.manual_seed(seed + 3)
    aux = torch.randint(-2**31, 2**31 - 1, (K * ld_aux,), generator=g, device="cuda", dtype=torch.int32)
    return dY, X, aux


def _oracle_abs_sum(oracle, dY, words, M, K, lda, ld_aux, dtype):
    dz, _ = oracle.drelu_bgrad(bits(dY), words, M, K, d_layout="col", ldd=lda, ld_aux=ld_aux, dtype=dtype)
    return np.abs(oracle.f16_decode(dz, dtype).reshape(K, lda)[:, :M]).sum(axis=0)


def run_dw(oracle, M, N, K, seed, dtype="f16", lda=None, ldx=None, ld_aux=None, want_bgrad=True):
    lda = lda or _pad8(M)
    ldx = ldx or _pad8(N)
    ld_aux = ld_aux or (M + 127) // 128 * 4
    ldd = _pad8(N)
    dY, X, aux = _inputs(M, N, K, seed, dtype, lda, ldx, ld_aux)
    L = ge.make_layout(MN, MN, ROW, lda, ldx, ldd, ld_aux)
    with ge.Plan(M, N, K, ge.GE_EPI_DW_DRELU_BGRAD, L, dtype=GE_DT[dtype]) as p:
        assert p.path == ge.GE_PATH_TC_GEMM
        cfg = p.config
        D = torch.full((M, ldd), float("nan"), dtype=TORCH_DTYPE[dtype], device="cuda")
        bgrad = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda") if want_bgrad else None
        p.execute(dY, X, bgrad, D, aux)
        torch.cuda.synchronize()
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
    words = aux.cpu().numpy().view(np.uint32)
    ref_dw, ref_bg = oracle.dw_drelu_bgrad(bits(dY), words, bits(X), M, N, K, lda=lda, ldb=ldx, ld_aux=ld_aux,
                                           dtype=dtype)
    what = f"dw_drelu {M}x{N}x{K} {dtype} cfg {cfg}"
    check_f16(oracle, bits(D[:, :N]), ref_dw, what, dtype)
    assert torch.isnan(D[:, N:].float()).all(), what + ": wrote past the columns"
    if want_bgrad:
        abs_sum = _oracle_abs_sum(oracle, dY, words, M, K, lda, ld_aux, dtype)
        check_bgrad(bgrad.cpu().numpy(), ref_bg, abs_sum, what + " bgrad")
    return cfg


@pytest.mark.parametrize("M,N,K", [(300, 264, 520), (129, 17, 72), (1000, 520, 1030), (64, 300, 4096)])
def test_dw_mask_shapes(oracle, M, N, K):
    """Ragged M (mask words and A rows past the end), ragged K (a partial last
    k-block), small and tall problems (the last splits K whole)."""
    run_dw(oracle, M, N, K, seed=600 + M)


def test_dw_mask_pitches_and_no_bgrad(oracle):
    run_dw(oracle, 300, 264, 520, seed=610, lda=320, ldx=272, ld_aux=16)
    run_dw(oracle, 300, 264, 520, seed=611, want_bgrad=False)


@pytest.mark.parametrize("tile_n,pair", [("128", "0"), ("256", "0"), ("256", "1")])
def test_dw_mask_tiles_and_split_tail(oracle, monkeypatch, tile_n, pair):
    monkeypatch.setenv("GE_TILE_N", tile_n)
    monkeypatch.setenv("GE_PAIR", pair)
    cfg = run_dw(oracle, 1000, 2056, 520, seed=620)
    assert cfg[1] == int(tile_n) and cfg[2] == int(pair)


def test_dw_mask_split_whole(oracle):
    """Under-filled problem: every tile split along K, bias-gradient pieces
    reduced in order."""
    cfg = run_dw(oracle, 256, 256, 2048, seed=630)
    assert cfg[3] > 1


def test_dw_mask_bf16(oracle):
    run_dw(oracle, 1000, 520, 1030, seed=640, dtype="bf16")


def test_dw_mask_matches_unfused_at_mlp_size(oracle):
    """dW[11008, 4096] over 8192 tokens: bit-identical to the standalone
    DRELU_BGRAD pass followed by the same GEMM on the stored dZ (the masked
    values are exact, and both GEMMs run the same tiles in the same order);
    sampled features against the oracle for dW rows and the bias gradient."""
    M, N, K = 11008, 4096, 8192
    ld_aux = (M + 127) // 128 * 4
    dY, X, aux = _inputs(M, N, K, 650, "f16", M, N, ld_aux)
    with ge.Plan(M, N, K, ge.GE_EPI_DW_DRELU_BGRAD, ge.make_layout(MN, MN, ROW)) as p:
        dW = torch.empty((M, N), dtype=torch.float16, device="cuda")
        bgrad = torch.empty(M, dtype=torch.float32, device="cuda")
        p.execute(dY, X, bgrad, dW, aux)
        torch.cuda.synchronize()
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
        cfg = p.config
    with ge.Plan(M, K, 0, ge.GE_EPI_DRELU_BGRAD, ge.make_layout(d=ge.GE_D_COL)) as pd, \
            ge.Plan(M, N, K, ge.GE_EPI_NONE, ge.make_layout(MN, MN, ROW)) as pg:
        assert pg.config == cfg
        dZ = torch.empty_like(dY)
        bg2 = torch.empty(M, dtype=torch.float32, device="cuda")
        pd.execute(dY, None, bg2, dZ, aux)
        dW2 = torch.empty_like(dW)
        pg.execute(dZ, X, None, dW2, None)
        torch.cuda.synchronize()
    assert torch.equal(dW.view(torch.int16), dW2.view(torch.int16)), "differs from DRELU_BGRAD + GEMM"
    assert torch.allclose(bgrad, bg2, rtol=1e-4, atol=1e-3)
    feats = sample_rows(M, 64, seed=0xD1)
    fi = torch.as_tensor(feats, device="cuda")
    words = aux.cpu().numpy().view(np.uint32).reshape(K, ld_aux)
    keep = np.unpackbits(words.view(np.uint8).reshape(K, -1), axis=1, bitorder="little")[:, feats]
    sub_words = np.packbits(np.concatenate([keep, np.zeros((K, 128 - len(feats)), np.uint8)], axis=1),
                            axis=1, bitorder="little").view(np.uint32)
    dY_sub = dY.index_select(1, fi).contiguous()
    ref_dw, ref_bg = oracle.dw_drelu_bgrad(bits(dY_sub), sub_words.reshape(-1), bits(X), len(feats), N, K,
                                           ld_aux=4)
    check_f16(oracle, bits(dW.index_select(0, fi)), ref_dw, "dw_drelu 11008x4096x8192 (features)")
    abs_sum = _oracle_abs_sum(oracle, dY_sub, sub_words.reshape(-1), len(feats), K, len(feats), 4, "f16")
    check_bgrad(bgrad.index_select(0, fi).cpu().numpy(), ref_bg, abs_sum, "dw_drelu bgrad (features)")
