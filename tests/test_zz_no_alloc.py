"""The allocation-free DRELU_BGRAD entry point (ge_drelu_bgrad_static).

It serves callers that cannot allocate device memory (its reduction scratch
is a fixed device array inside the library). Its results must match the
plan-based DRELU_BGRAD (which allocates a plan workspace) and the fp64
oracle within the tests' tolerances, on consecutive calls that share the
scratch, also when the problem needs more row splits than the scratch holds
(the call then uses fewer), and a call must leave the device's free memory
unchanged. This file is collected last so a failure here never hides the
other tests' results.
"""
import numpy as np
import pytest
import torch

import gemm_epilogues_gb300 as ge
from gemm_epilogues_gb300.inputs import f16_tensor

from _util import bits, check_bgrad

pytestmark = pytest.mark.gpu


def _mask_for(M, N, d, seed):
    """A forward RELU_AUX_BIAS mask for an [M, N] problem stored in layout d."""
    K = 64
    dl = ge.GE_D_ROW if d == "row" else ge.GE_D_COL
    W = f16_tensor((M, K), seed + 1).cuda()
    X = f16_tensor((N, K), seed + 2).cuda()
    b = f16_tensor((M,), seed + 3).cuda()
    with ge.Plan(M, N, K, ge.GE_EPI_RELU_AUX_BIAS, ge.make_layout(ge.GE_K_MAJOR, ge.GE_K_MAJOR, dl)) as p:
        rows, cols = (M, N) if d == "row" else (N, M)
        Y = torch.empty((rows, cols), dtype=torch.float16, device="cuda")
        aux = torch.empty(p.aux_bytes // 4, dtype=torch.int32, device="cuda")
        p.execute(W, X, b, Y, aux)
        torch.cuda.synchronize()
        return aux, p.aux_ld


def _plan_drelu(M, N, d, dY, aux):
    dl = ge.GE_D_ROW if d == "row" else ge.GE_D_COL
    with ge.Plan(M, N, 0, ge.GE_EPI_DRELU_BGRAD, ge.make_layout(d=dl)) as p:
        dZ = torch.empty_like(dY)
        bg = torch.empty(M, dtype=torch.float32, device="cuda")
        p.execute(dY, None, bg, dZ, aux)
        torch.cuda.synchronize()
    return dZ, bg


def _static(M, N, d, ld_aux, dY, aux):
    dZ = torch.full_like(dY, float("nan"))
    bg = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
    dl = ge.GE_D_ROW if d == "row" else ge.GE_D_COL
    ge.ge_drelu_bgrad_static(M, N, dl, 0, ld_aux, dY, aux, dZ, bg)
    torch.cuda.synchronize()
    return dZ, bg


def _check_oracle(oracle, M, N, d, ld_aux, dY, aux, dZ, bg, what):
    """dZ bit-exact and the bias gradient within the 1e-4 bounds, against the
    fp64 oracle on the same bits."""
    rdz, rbg = oracle.drelu_bgrad(bits(dY), aux.cpu().numpy().view(np.uint32), M, N, d_layout=d, ld_aux=ld_aux)
    assert np.array_equal(bits(dZ), rdz), f"{what}: dZ differs from the oracle"
    rows, cols = (M, N) if d == "row" else (N, M)
    abs_sum = np.abs(oracle.f16_decode(rdz).reshape(rows, cols)).sum(axis=1 if d == "row" else 0)
    check_bgrad(bg.cpu().numpy(), rbg, abs_sum, what)


def _compare_plan(dZ_s, bg_s, dZ_p, bg_p, d):
    assert torch.equal(dZ_s.view(torch.int16), dZ_p.view(torch.int16)), "dZ differs from the plan's"
    dzf = dZ_p.float().cpu().numpy().astype(np.float64)
    abs_sum = np.abs(dzf).sum(axis=0 if d == "col" else 1)
    a = bg_s.cpu().numpy().astype(np.float64)
    b = bg_p.cpu().numpy().astype(np.float64)
    tol = 1e-4 * np.maximum(np.abs(b), abs_sum * 2.0 ** -7)
    assert (np.abs(a - b) <= tol).all(), f"bgrad differs from the plan's (worst {np.abs(a - b).max():.3g})"


@pytest.mark.parametrize("d", ["col", "row"])
def test_static_matches_plan_and_oracle_on_two_calls(oracle, d):
    problems = [(11008, 1024, 71), (3000, 776, 72)]  # the second reuses the scratch
    for M, N, seed in problems:
        aux, ld_aux = _mask_for(M, N, d, seed * 10)
        rows, cols = (M, N) if d == "row" else (N, M)
        dY = f16_tensor((rows, cols), seed * 10 + 4).cuda()
        dZ_p, bg_p = _plan_drelu(M, N, d, dY, aux)
        dZ_s, bg_s = _static(M, N, d, ld_aux, dY, aux)
        _compare_plan(dZ_s, bg_s, dZ_p, bg_p, d)
        _check_oracle(oracle, M, N, d, ld_aux, dY, aux, dZ_s, bg_s, f"static {d} {M}x{N}")


def test_static_fewer_splits_than_asked_matches_oracle(oracle, monkeypatch):
    # 16384 features x 4352 tokens, column layout: 68 row splits are asked for
    # (GE_DRELU_SPLITS, read at every call), but 68 x 16384 x 4 bytes of
    # partial sums exceed the 4 MiB scratch, so the call runs 63 splits. The
    # sums then take another order than the plan's; both stay within the
    # bound against the oracle.
    M, N = 16384, 4352
    d = "col"
    ld_aux = (M + 127) // 128 * 4
    dY = f16_tensor((N, M), 7301).cuda()
    g = torch.Generator(device="cuda")
    g.manual_seed(7302)
    aux = torch.randint(-2**31, 2**31 - 1, (N * ld_aux,), generator=g, device="cuda", dtype=torch.int32)
    monkeypatch.setenv("GE_DRELU_SPLITS", "256")
    for _ in range(2):  # two calls in a row on the shared scratch
        dZ, bg = _static(M, N, d, ld_aux, dY, aux)
        _check_oracle(oracle, M, N, d, ld_aux, dY, aux, dZ, bg, "static, splits cut to fit the scratch")


def test_static_call_allocates_nothing():
    M, N = 11008, 2048
    aux, ld_aux = _mask_for(M, N, "col", 740)
    dY = f16_tensor((N, M), 744).cuda()
    dZ = torch.empty_like(dY)
    bg = torch.empty(M, dtype=torch.float32, device="cuda")
    # the first call on this device may load the library's kernels and look
    # up the scratch address; what follows must not allocate
    ge.ge_drelu_bgrad_static(M, N, ge.GE_D_COL, 0, ld_aux, dY, aux, dZ, bg)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(2):
        ge.ge_drelu_bgrad_static(M, N, ge.GE_D_COL, 0, ld_aux, dY, aux, dZ, bg)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert torch.cuda.memory_allocated() == alloc0


def test_static_rejects_beyond_scratch():
    # A column-major problem whose partial sums cannot fit in the fixed
    # scratch is refused before anything is launched.
    t = torch.zeros(64, dtype=torch.float16, device="cuda")
    aux = torch.zeros(64, dtype=torch.int32, device="cuda")
    bg = torch.zeros(64, dtype=torch.float32, device="cuda")
    M = 2_000_000
    st = ge.ge_drelu_bgrad_static(M, 8, ge.GE_D_COL, 0, 0, t, aux, t, bg, raw=True)
    assert st == ge.GE_ERR_UNSUPPORTED
    assert ge.ge_drelu_bgrad_static(8, 8, ge.GE_D_COL, 0, 0, None, aux, t, bg, raw=True) == ge.GE_ERR_INVALID_ARG
