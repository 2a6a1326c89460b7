"""The workloads at full size, in the launch configuration the benchmark
times: outputs checked against the oracle on sampled stored rows (256 per
problem, or all rows where the oracle is quick), plus properties that hold at
any size (finite outputs, mask consistent with the stored values)."""
import numpy as np
import pytest
import torch

import gemm_epilogues_gb300 as ge
from gemm_epilogues_gb300.inputs import pages_workloads, sample_rows

from _util import bits, check_bgrad, check_f16, check_mask, gpu_forward, oracle_full, oracle_rows

pytestmark = pytest.mark.gpu

W = pages_workloads()


def _check_sampled(oracle, w, A, B, bias, D, aux, ld_aux, rows=None):
    d_rows, d_cols = w.d_shape()
    rows = sample_rows(d_rows) if rows is None else rows
    ref = oracle_rows(oracle, w, A, B, bias, rows)
    idx = torch.as_tensor(rows, device=D.device)
    got = bits(D.index_select(0, idx))
    check_f16(oracle, got, ref["D"], w.name)
    if aux is not None:
        gw = aux.view(d_rows, ld_aux).index_select(0, idx).cpu().numpy().view(np.uint32).reshape(-1)
        check_mask(gw, ref["aux"], ref["Z"], len(rows), d_cols, ld_aux, w.name)


def _make_gpu(w):
    return w.make("cuda")


@pytest.mark.parametrize("key", ["c3_T1", "c3_T512", "c3_T2048"])
def test_ffn_up_gelu(oracle, key):
    w = W[key]
    A, B, bias = _make_gpu(w)
    D, aux, path, ld_aux = gpu_forward(w, A, B, bias)
    assert path == (ge.GE_PATH_GEMV if w.N <= 16 else ge.GE_PATH_TC_GEMM)
    if w.N <= 512:
        ref = oracle_full(oracle, w, A.cpu(), B.cpu(), bias.cpu())
        check_f16(oracle, bits(D), ref["D"], w.name)
    else:
        _check_sampled(oracle, w, A, B, bias, D, None, 0)


def test_mlp_training_pair(oracle):
    """Forward RELU_AUX_BIAS, DRELU_BGRAD on dY, then the dW GEMM, at the
    LLaMA-7B MLP size; each stage against the oracle."""
    w = W["c4_fwd"]
    A, B, bias = _make_gpu(w)
    D, aux, path, ld_aux = gpu_forward(w, A, B, bias)
    assert path == ge.GE_PATH_TC_GEMM
    _check_sampled(oracle, w, A, B, bias, D, aux, ld_aux)
    # whole-tensor properties: finite, ReLU outputs non-negative
    assert torch.isfinite(D.float()).all()
    assert (D >= 0).all()
    # backward
    T, O = w.N, w.M
    dY = torch.empty((T, O), dtype=torch.float16, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(3004)
    dY.copy_(torch.randn((T, O), generator=g, device="cuda"))
    L = ge.make_layout(d=ge.GE_D_COL)
    with ge.Plan(O, T, 0, ge.GE_EPI_DRELU_BGRAD, L) as p:
        dZ = torch.empty_like(dY)
        bgrad = torch.empty(O, dtype=torch.float32, device="cuda")
        p.execute(dY, None, bgrad, dZ, aux)
        torch.cuda.synchronize()
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
    ref_dz, ref_bg = oracle.drelu_bgrad(bits(dY), aux.cpu().numpy().view(np.uint32), O, T,
                                        d_layout="col", ld_aux=ld_aux)
    assert np.array_equal(bits(dZ), ref_dz)
    abs_sum = np.abs(oracle.f16_decode(ref_dz).reshape(T, O)).sum(axis=0)
    check_bgrad(bgrad.cpu().numpy(), ref_bg, abs_sum, "c4 bwd")
    # dW = dZ^T . X  (A = dZ read M-major, B = X read N-major, D row-major)
    wd = W["c4_dw"]
    zero_bias = torch.zeros(wd.M, dtype=torch.float16, device="cuda")  # unused by NONE
    Dw, _, path, _ = gpu_forward(wd, dZ, B, zero_bias)
    assert path == ge.GE_PATH_TC_GEMM
    _check_sampled(oracle, wd, dZ, B, zero_bias, Dw, None, 0)


def test_large_relu_aux(oracle):
    w = W["c5"]
    A, B, bias = _make_gpu(w)
    D, aux, path, ld_aux = gpu_forward(w, A, B, bias)
    assert path == ge.GE_PATH_TC_GEMM
    _check_sampled(oracle, w, A, B, bias, D, aux, ld_aux)
    assert torch.isfinite(D.float()).all()
    assert (D >= 0).all()
