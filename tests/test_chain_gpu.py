"""A stack of decode projections in one launch (ge_execute_chain) against
the oracle: every layer's stored output is checked against the oracle's
forward applied to that layer's weights and bias and to the GPU's own stored
input of the layer (the previous layer's output), within the 16-bit output
tolerance. Ragged row counts per block, fewer rows than blocks, several
tokens, bf16, no bias, repeated launches (the synchronisation words are
reused) and the argument checks."""
import numpy as np
import pytest
import torch

import gemm_epilogues_gb300 as ge
from gemm_epilogues_gb300.inputs import TORCH_DTYPE, f16_tensor

from _util import GE_DT, bits, check_f16

pytestmark = pytest.mark.gpu

KK = ge.GE_K_MAJOR


def _layers(M, L, epi, seed, dtype):
    t = TORCH_DTYPE[dtype]
    Ws = [f16_tensor((M, M), seed + 10 * l, "normal", 1.0 / np.sqrt(M), "cuda", t) for l in range(L)]
    bs = None if epi == "none" else [f16_tensor((M,), seed + 10 * l + 1, "normal", 0.1, "cuda", t)
                                     for l in range(L)]
    return Ws, bs


def run_chain(oracle, M, N, L, epi, seed, dtype="f16"):
    t = TORCH_DTYPE[dtype]
    Ws, bs = _layers(M, L, epi, seed, dtype)
    X = f16_tensor((N, M), seed + 7, "normal", 1.0, "cuda", t)
    Y = torch.full((L, N, M), float("nan"), dtype=t, device="cuda")
    with ge.Plan(M, N, M, ge.EPILOGUE_BY_NAME[epi], ge.make_layout(KK, KK, ge.GE_D_COL), dtype=GE_DT[dtype]) as p:
        p.execute_chain(Ws, bs, X, Y)
        torch.cuda.synchronize()
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
    prev = X
    for l in range(L):
        ref = oracle.linear_forward(bits(Ws[l]), bits(prev), None if bs is None else bits(bs[l]), epi, M, N, M,
                                    a_major="k", b_major="k", d_layout="col", dtype=dtype)
        check_f16(oracle, bits(Y[l]), ref["D"], f"chain layer {l} of {L} ({M}x{N}, {epi}, {dtype})", dtype)
        prev = Y[l]
    return Ws, bs, X, Y


@pytest.mark.parametrize("M,N,L,epi", [
    (256, 1, 3, "gelu_bias"),      # fewer rows than warps: most warps idle
    (64, 2, 3, "relu_bias"),       # fewer rows than blocks: most blocks idle
    (1000, 3, 5, "relu_bias"),     # ragged rows per block and per warp
    (520, 16, 2, "bias"),          # the widest token count
    (384, 5, 4, "none"),           # no bias
    (2048, 1, 6, "gelu_erf_bias"),
    (4096, 16, 2, "gelu_bias"),    # 16 tokens: whole-row items, a ring of 12 slots for 27 rows a block
    (2048, 4, 3, "relu_bias"),     # four tokens: half-row items, the ring longer than a layer
    (4864, 1, 3, "gelu_bias"),     # 32 rows a block: half-row items, the ring shorter than a layer
    (4864, 4, 2, "bias"),
])
def test_chain_matches_oracle_per_layer(oracle, M, N, L, epi):
    run_chain(oracle, M, N, L, epi, seed=9000 + M + 31 * N)


@pytest.mark.parametrize("N", [1, 2])
def test_chain_bf16(oracle, N):
    run_chain(oracle, 776, N, 3, "gelu_bias", seed=9100 + N, dtype="bf16")


def test_chain_one_token_longer_rows(oracle):
    """K = 6144: one layer of a block's rows (41 rows of 12 KB) does not fit
    in shared memory, so each warp streams through a ring of a few half
    rows."""
    run_chain(oracle, 6144, 1, 3, "gelu_bias", seed=9150)


def test_chain_decode_size(oracle):
    """Eight 4096 x 4096 layers, one token."""
    run_chain(oracle, 4096, 1, 8, "gelu_bias", seed=9200)


def test_chain_benchmark_stack(oracle):
    """The benchmark's decode stack as it is timed: 32 layers of 4096 x 4096
    fp16 (weights N(0, 1/64^2), biases N(0, 0.02)), one token, every layer
    against the oracle on its stored input."""
    M, L = 4096, 32
    Ws = [f16_tensor((M, M), 2200 + i, "normal", 1 / 64, "cuda") for i in range(L)]
    bs = [f16_tensor((M,), 2300 + i, "normal", 0.02 ** 0.5, "cuda") for i in range(L)]
    X = f16_tensor((1, M), 2002, "normal", 1.0, "cuda")
    Y = torch.full((L, 1, M), float("nan"), dtype=torch.float16, device="cuda")
    with ge.Plan(M, 1, M, ge.GE_EPI_GELU_BIAS, ge.make_layout(KK, KK, ge.GE_D_COL)) as p:
        p.execute_chain(Ws, bs, X, Y)
        torch.cuda.synchronize()
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
    prev = X
    for l in range(L):
        ref = oracle.linear_forward(bits(Ws[l]), bits(prev), bits(bs[l]), "gelu_bias", M, 1, M,
                                    a_major="k", b_major="k", d_layout="col")
        check_f16(oracle, bits(Y[l]), ref["D"], f"benchmark stack layer {l}")
        prev = Y[l]


def test_chain_full_depth_and_repeat(oracle):
    """64 layers (the limit) twice in a row: the second launch waits for its
    own layers' tagged exchange words, not the first launch's; both launches
    give the same bits, and the last layer still matches the oracle on its
    stored input."""
    M, N, L = 512, 1, 64
    Ws, bs = _layers(M, L, "gelu_bias", 9300, "f16")
    X = f16_tensor((N, M), 9399, "normal", 1.0, "cuda")
    Y1 = torch.empty((L, N, M), dtype=torch.float16, device="cuda")
    Y2 = torch.empty_like(Y1)
    with ge.Plan(M, N, M, ge.GE_EPI_GELU_BIAS, ge.make_layout(KK, KK, ge.GE_D_COL)) as p:
        p.execute_chain(Ws, bs, X, Y1)
        p.execute_chain(Ws, bs, X, Y2)
        torch.cuda.synchronize()
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    ref = oracle.linear_forward(bits(Ws[-1]), bits(Y1[-2]), bits(bs[-1]), "gelu_bias", M, N, M,
                                a_major="k", b_major="k", d_layout="col")
    check_f16(oracle, bits(Y1[-1]), ref["D"], "layer 64")


def test_chain_depths_in_turn_on_one_plan(oracle):
    """One plan running chains of 3, 1, 2, 5, 1, 3 layers in turn, each with
    new weights and input: the exchange words a launch leaves behind (its
    tags, in both halves of the exchange) never pass for the next launch's,
    whatever the depths; every layer of every launch against the oracle."""
    M, N = 776, 2
    with ge.Plan(M, N, M, ge.GE_EPI_RELU_BIAS, ge.make_layout(KK, KK, ge.GE_D_COL)) as p:
        for r, L in enumerate((3, 1, 2, 5, 1, 3)):
            Ws, bs = _layers(M, L, "relu_bias", 9500 + 100 * r, "f16")
            X = f16_tensor((N, M), 9550 + 100 * r, "normal", 1.0, "cuda")
            Y = torch.full((L, N, M), float("nan"), dtype=torch.float16, device="cuda")
            p.execute_chain(Ws, bs, X, Y)
            torch.cuda.synchronize()
            assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
            prev = X
            for l in range(L):
                ref = oracle.linear_forward(bits(Ws[l]), bits(prev), bits(bs[l]), "relu_bias", M, N, M,
                                            a_major="k", b_major="k", d_layout="col")
                check_f16(oracle, bits(Y[l]), ref["D"], f"launch {r} layer {l} of {L}")
                prev = Y[l]


def test_chain_in_a_cuda_graph(oracle):
    """A 3-layer chain captured in a CUDA graph and replayed with new inputs
    copied into the captured buffer: each replay advances the launch epoch
    on the device, so its layers never take the previous replay's exchange
    words; every replay bit-identical to an eager launch on the same input."""
    M, N, L = 1000, 2, 3
    Ws, bs = _layers(M, L, "gelu_bias", 9600, "f16")
    X = torch.empty((N, M), dtype=torch.float16, device="cuda")
    Y = torch.empty((L, N, M), dtype=torch.float16, device="cuda")
    with ge.Plan(M, N, M, ge.GE_EPI_GELU_BIAS, ge.make_layout(KK, KK, ge.GE_D_COL)) as p:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            X.copy_(f16_tensor((N, M), 9601, "normal", 1.0, "cuda"))
            p.execute_chain(Ws, bs, X, Y, s)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            p.execute_chain(Ws, bs, X, Y, torch.cuda.current_stream())
        for r in range(3):
            Xr = f16_tensor((N, M), 9610 + r, "normal", 1.0, "cuda")
            X.copy_(Xr)
            Y.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
            Ye = torch.full_like(Y, float("nan"))
            p.execute_chain(Ws, bs, Xr, Ye)
            torch.cuda.synchronize()
            assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
            assert torch.equal(Y.view(torch.int16), Ye.view(torch.int16)), f"replay {r}"
            ref = oracle.linear_forward(bits(Ws[0]), bits(Xr), bits(bs[0]), "gelu_bias", M, N, M,
                                        a_major="k", b_major="k", d_layout="col")
            check_f16(oracle, bits(Y[0]), ref["D"], f"replay {r} layer 0")


def test_chain_first_layer_equals_single_gemv(oracle):
    """Layer 0 of a chain against the single-layer decode GEMV on the same
    inputs: both within the tolerance of the oracle and of each other."""
    M, N = 4096, 1
    Ws, bs = _layers(M, 2, "gelu_bias", 9400, "f16")
    X = f16_tensor((N, M), 9401, "normal", 1.0, "cuda")
    Y = torch.empty((2, N, M), dtype=torch.float16, device="cuda")
    y1 = torch.empty((N, M), dtype=torch.float16, device="cuda")
    with ge.Plan(M, N, M, ge.GE_EPI_GELU_BIAS, ge.make_layout(KK, KK, ge.GE_D_COL)) as p:
        p.execute_chain(Ws, bs, X, Y)
        p.execute(Ws[0], X, bs[0], y1)
        torch.cuda.synchronize()
    check_f16(oracle, bits(Y[0]), bits(y1), "chain layer 0 vs GEMV")


def test_chain_rejects():
    M = 256
    W = torch.zeros((M, M), dtype=torch.float16, device="cuda")
    b = torch.zeros(M, dtype=torch.float16, device="cuda")
    X = torch.zeros((1, M), dtype=torch.float16, device="cuda")
    Y = torch.zeros((2, 1, M), dtype=torch.float16, device="cuda")
    col = ge.make_layout(KK, KK, ge.GE_D_COL)
    with ge.Plan(M, 1, M, ge.GE_EPI_BIAS, col) as p:
        run = lambda *a: ge.ge_execute_chain(p.handle, *a, raw=True)
        assert run([W, W], [b, b], X, Y) == ge.GE_OK
        assert run([], [], X, Y) == ge.GE_ERR_INVALID_ARG
        assert run([W] * 65, [b] * 65, X, Y) == ge.GE_ERR_INVALID_ARG
        assert run([W, None], [b, b], X, Y) == ge.GE_ERR_INVALID_ARG
        assert run([W, W], None, X, Y) == ge.GE_ERR_INVALID_ARG  # BIAS needs biases
        assert run([W, W], [b, b], None, Y) == ge.GE_ERR_INVALID_ARG
        Xo = torch.zeros(M + 8, dtype=torch.float16, device="cuda")[1:M + 1]  # 2 bytes off 16
        assert run([W, W], [b, b], Xo, Y) == ge.GE_ERR_ALIGNMENT
        assert run([W, W], [b, b], X, torch.zeros(4, device="cpu")) == ge.GE_ERR_DEVICE_MISMATCH
        torch.cuda.synchronize()
    with ge.Plan(M, 1, M + 8, ge.GE_EPI_BIAS, col) as p:  # not square
        assert ge.ge_execute_chain(p.handle, [W], [b], X, Y, raw=True) == ge.GE_ERR_UNSUPPORTED
    with ge.Plan(M, 1, M, ge.GE_EPI_BIAS, ge.make_layout(KK, KK, ge.GE_D_ROW)) as p:  # D row-major
        assert ge.ge_execute_chain(p.handle, [W], [b], X, Y, raw=True) == ge.GE_ERR_UNSUPPORTED
    with ge.Plan(M, 32, M, ge.GE_EPI_BIAS, col) as p:  # tensor-core path
        assert ge.ge_execute_chain(p.handle, [W], [b], X, Y, raw=True) == ge.GE_ERR_UNSUPPORTED


@pytest.mark.parametrize("producers", ["1", "2"])
@pytest.mark.parametrize("M,N,L,epi", [
    (4096, 1, 4, "gelu_bias"),
    (6144, 1, 2, "gelu_bias"),     # the ring shorter than a layer: slots shared by several warps' items
    (1000, 3, 5, "relu_bias"),
    (520, 16, 2, "bias"),
])
def test_chain_producer_warps(oracle, monkeypatch, producers, M, N, L, epi):
    """One, two or 32 producer lanes sharing out a block's bulk copies (by
    default the count from 8 to 32 that keeps the most ring slots): the
    ring's slots cut to a multiple of their number."""
    monkeypatch.setenv("GE_CHAIN_PRODUCERS", producers)
    run_chain(oracle, M, N, L, epi, seed=9300 + M + 31 * N)
