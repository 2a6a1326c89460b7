"""Parity of the DRELU_BGRAD kernel (mask applied to dY, fp32 bias gradient)
with the CPU oracle, both storage layouts, ragged extents, repeated calls."""
import numpy as np
import pytest
import torch

import gemm_epilogues_gb300 as ge
from gemm_epilogues_gb300.inputs import TORCH_DTYPE, Workload, f16_tensor

from _util import GE_DT, bits, check_bgrad, gpu_forward, oracle_full

pytestmark = pytest.mark.gpu


def _pad8(x):
    return (x + 7) // 8 * 8


def run_drelu(oracle, M, N, dl, seed, inplace=False, repeat=1, dtype="f16"):
    K = 72
    t = TORCH_DTYPE[dtype]
    w = Workload("fwd", M, N, K, "relu_aux_bias", "k", "k" if dl == "col" else "n", dl, dtype=dtype)
    rows, cols = w.d_shape()
    ldd = _pad8(cols)
    b_rows, b_cols = w.b_shape()
    ldb = _pad8(b_cols)
    A = f16_tensor(w.a_shape(), seed + 1, dtype=t).cuda()
    B = f16_tensor((b_rows, ldb), seed + 2, dtype=t).cuda()
    bias = f16_tensor((M,), seed + 3, dtype=t).cuda()
    _, aux, _, ld_aux = gpu_forward(w, A, B, bias, ld=dict(ldb=ldb, ldd=ldd))
    dY = f16_tensor((rows, ldd), seed + 4, "normal", 2.0, dtype=t).cuda()
    dY_host = dY.cpu()
    L = ge.make_layout(d=ge.GE_D_ROW if dl == "row" else ge.GE_D_COL, ldd=ldd)
    with ge.Plan(M, N, 0, ge.GE_EPI_DRELU_BGRAD, L, dtype=GE_DT[dtype]) as p:
        assert p.path == ge.GE_PATH_DRELU
        dZ = dY if inplace else torch.full_like(dY, float("nan"))
        bgrad = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
        for _ in range(repeat):
            if inplace:
                dZ.copy_(dY_host.cuda())
            p.execute(dY if not inplace else dZ, None, bgrad, dZ, aux)
        torch.cuda.synchronize()
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
    ref_dz, ref_bg = oracle.drelu_bgrad(bits(dY_host), aux.cpu().numpy().view(np.uint32), M, N,
                                        d_layout=dl, ldd=ldd, ld_aux=ld_aux, dtype=dtype)
    got = bits(dZ).reshape(rows, ldd)[:, :cols]
    assert np.array_equal(got, ref_dz.reshape(rows, ldd)[:, :cols]), "dZ not bit-identical"
    dzf = oracle.f16_decode(ref_dz, dtype).reshape(rows, ldd)[:, :cols]
    abs_sum = np.abs(dzf).sum(axis=0 if dl == "col" else 1)
    check_bgrad(bgrad.cpu().numpy(), ref_bg, abs_sum, f"drelu {M}x{N} {dl}")
    return bgrad


@pytest.mark.parametrize("M,N", [(1, 1), (37, 5), (256, 256), (300, 1000), (1000, 300), (2050, 129)])
@pytest.mark.parametrize("dl", ["row", "col"])
def test_drelu_shapes(oracle, M, N, dl):
    run_drelu(oracle, M, N, dl, seed=100 + M + N)


@pytest.mark.parametrize("dl", ["row", "col"])
def test_drelu_inplace_and_repeat(oracle, dl):
    """dZ may alias dY, and the workspace counters reset between calls."""
    run_drelu(oracle, 777, 2333, dl, seed=5, inplace=True, repeat=3)


def test_drelu_deterministic(oracle):
    b1 = run_drelu(oracle, 1500, 4000, "col", seed=9)
    b2 = run_drelu(oracle, 1500, 4000, "col", seed=9)
    assert torch.equal(b1, b2)
