"""bfloat16 operands, bias and output (fp32 accumulation) through every
kernel: the tensor-core GEMM in each operand major and D layout, 2-SM tiles,
the split-K tail, the GEMV, the unfused baseline, DRELU_BGRAD standalone and
as a GEMM epilogue. Each result is compared with the oracle run on the same
bf16 bit patterns (the oracle decodes and rounds bf16 itself)."""
import itertools

import numpy as np
import pytest
import torch

import gemm_epilogues_gb300 as ge

from test_drelu_gpu import run_drelu
from test_gemm_drelu_gpu import run_case as run_gemm_drelu
from test_gemm_gpu import EPIS, _run_case

pytestmark = pytest.mark.gpu

BF = "bf16"


@pytest.mark.parametrize("am,bm,dl", list(itertools.product("km", "kn", ("row", "col"))))
def test_bf16_layouts_ragged(oracle, am, bm, dl):
    for i, (M, N, K) in enumerate([(300, 520, 200), (129, 257, 72)]):
        epi = EPIS[(M + N + K + i) % len(EPIS)]
        path = _run_case(oracle, M, N, K, epi, am, bm, dl, seed=200 + i, dtype=BF)
        assert path == ge.GE_PATH_TC_GEMM


@pytest.mark.parametrize("epi", EPIS + ["gelu_erf_bias"])
def test_bf16_every_epilogue(oracle, epi):
    _run_case(oracle, 1024, 512, 2048, epi, "k", "n", "row", dist=("normal", 2048 ** -0.5), seed=210,
              dtype=BF)


@pytest.mark.parametrize("epi", ["none", "bias", "relu_bias", "relu_aux_bias"])
def test_bf16_exact_integer(oracle, epi):
    """Integers in [-1, 1] with K = 128 and a bias in [-8, 8]: every sum has at
    most 8 significant bits, so it is exact in bf16 and the result is
    bit-identical (the mask too)."""
    _run_case(oracle, 256, 264, 128, epi, "k", "n", "row", dist=("int", 1.0), seed=220, exact=True,
              dtype=BF)
    _run_case(oracle, 256, 264, 128, epi, "m", "k", "col", dist=("int", 1.0), seed=221, exact=True,
              dtype=BF)


@pytest.mark.parametrize("epi", ["bias", "relu_aux_bias", "gelu_bias"])
def test_bf16_pair_tiles_and_split_tail(oracle, monkeypatch, epi):
    monkeypatch.setenv("GE_PAIR", "1")
    monkeypatch.setenv("GE_TILE_N", "256")
    _run_case(oracle, 1000, 2056, 520, epi, "k", "n", "row", seed=230, dtype=BF)
    _run_case(oracle, 513, 264, 4100, epi, "m", "k", "col", seed=231, dtype=BF)


@pytest.mark.parametrize("N", [1, 3, 16])
@pytest.mark.parametrize("epi", ["none", "bias", "relu_bias", "gelu_bias", "gelu_erf_bias"])
def test_bf16_gemv(oracle, N, epi):
    path = _run_case(oracle, 1000, N, 1030, epi, "k", "k", "col", seed=240 + N, dtype=BF)
    assert path == (ge.GE_PATH_GEMV if N <= 4 else ge.GE_PATH_TC_GEMM)


@pytest.mark.parametrize("epi", ["bias", "relu_bias", "gelu_bias", "relu_aux_bias"])
def test_bf16_unfused(oracle, epi):
    _run_case(oracle, 300, 520, 200, epi, "k", "n", "row", seed=250, unfused=True, dtype=BF)
    _run_case(oracle, 300, 517, 200, epi, "k", "k", "col", seed=251, unfused=True, dtype=BF)


@pytest.mark.parametrize("M,N", [(37, 5), (300, 1000), (2050, 129)])
@pytest.mark.parametrize("dl", ["row", "col"])
def test_bf16_drelu_standalone(oracle, M, N, dl):
    run_drelu(oracle, M, N, dl, seed=260 + M, dtype=BF)


def test_bf16_drelu_inplace(oracle):
    run_drelu(oracle, 777, 2333, "col", seed=265, inplace=True, repeat=2, dtype=BF)


@pytest.mark.parametrize("am,bm,dl", [("k", "n", "row"), ("k", "k", "col"), ("m", "n", "row"), ("m", "k", "col")])
def test_bf16_gemm_drelu_bgrad(oracle, am, bm, dl):
    run_gemm_drelu(oracle, 300, 520, 200, am, bm, dl, seed=270, dtype=BF)
    run_gemm_drelu(oracle, 257, 129, 1030, am, bm, dl, seed=271, dtype=BF)


def test_bf16_gemm_drelu_bgrad_exact_integer(oracle):
    run_gemm_drelu(oracle, 264, 520, 128, "k", "n", "row", seed=275, dist=("int", 1.0), exact=True,
                   dtype=BF)

