"""Parity of the tcgen05 GEMM + fused epilogue (and the GEMV path) with the
CPU oracle, element by element, on small and odd shapes in every layout."""
import itertools

import numpy as np
import pytest
import torch

import gemm_epilogues_gb300 as ge
from gemm_epilogues_gb300.inputs import TORCH_DTYPE, Workload, f16_tensor

from _util import (MASK_BAND, bits, check_f16, check_mask, gpu_forward, oracle_full)

pytestmark = pytest.mark.gpu

EPIS = ["none", "bias", "relu_bias", "gelu_bias", "relu_aux_bias"]


def _pad8(x):
    return (x + 7) // 8 * 8


def _run_case(oracle, M, N, K, epi, am, bm, dl, dist=("normal", 1.0), seed=0, exact=False,
              unfused=False, dtype="f16"):
    w = Workload(f"{M}x{N}x{K} {epi} {am}{bm}{dl} {dtype}", M, N, K, epi, am, bm, dl,
                 a_dist=dist, b_dist=dist, bias_dist=(dist[0], 4.0 if dist[0] == "int" else 1.0),
                 dtype=dtype)
    t = TORCH_DTYPE[dtype]
    # storage with padded leading dimensions (multiples of 8 elements)
    a_rows, a_cols = w.a_shape()
    b_rows, b_cols = w.b_shape()
    d_rows, d_cols = w.d_shape()
    lda, ldb, ldd = _pad8(a_cols), _pad8(b_cols), _pad8(d_cols)
    g = seed * 10
    Ap = f16_tensor((a_rows, lda), g + 1, *dist, dtype=t).cuda()
    Bp = f16_tensor((b_rows, ldb), g + 2, *dist, dtype=t).cuda()
    if dist[0] == "int":
        bias = f16_tensor((M,), g + 3, "int", 8, dtype=t).cuda()
    else:
        bias = f16_tensor((M,), g + 3, *dist, dtype=t).cuda()
    # poison the padding so a read past the logical extent shows up
    Ap[:, a_cols:] = float("nan")
    Bp[:, b_cols:] = float("nan")
    ld = dict(lda=lda, ldb=ldb, ldd=ldd)
    D, aux, path, ld_aux = gpu_forward(w, Ap, Bp, bias, unfused=unfused, ld=ld)
    ref = oracle_full(oracle, w, Ap.cpu(), Bp.cpu(), bias.cpu(), ld=ld)
    got = bits(D).reshape(d_rows, ldd)[:, :d_cols].reshape(-1)
    want = ref["D"].reshape(d_rows, ldd)[:, :d_cols].reshape(-1)
    extra = None
    mask_band = None
    if unfused and dtype == "bf16" and epi != "none":
        # The unfused flow stores A.B rounded to bf16 before adding the bias:
        # where the bias cancels most of A.B, that rounding (up to half a
        # bf16 step of |A.B|, 2^-9 |A.B|) is large next to the result. Allow
        # it, doubled for the activation's slope (at most 1.13 for GELU).
        Z = ref["Z"].reshape(d_rows, ldd)[:, :d_cols]
        bias64 = oracle.f16_decode(bits(bias).reshape(-1), dtype)
        bz = bias64[:, None] if dl == "row" else bias64[None, :]
        extra = 2.0 ** -8 * np.abs(Z - bz)
        # the mask comes from the rounded z too: a sign can flip within it
        mask_band = MASK_BAND + extra
        extra = extra.reshape(-1)
    if exact:
        assert np.array_equal(got, want), f"{w.name}: not bit-identical"
    else:
        check_f16(oracle, got, want, w.name, dtype, extra_tol=extra)
    # padding columns of D are never written
    padv = D[:, d_cols:]
    assert torch.isnan(padv.float()).all(), f"{w.name}: wrote past the logical columns"
    if epi == "relu_aux_bias":
        assert ld_aux == ref["ld_aux"]
        Z = ref["Z"].reshape(d_rows, ldd)[:, :d_cols]
        gw = aux.cpu().numpy().view(np.uint32)
        if exact:
            assert np.array_equal(gw, ref["aux"]), f"{w.name}: mask not bit-identical"
        else:
            check_mask(gw, ref["aux"], Z, d_rows, d_cols, ld_aux, w.name, band=mask_band)
    return path


def test_config1_bias(oracle):
    """256x128x512 BIAS, uniform [0,1) data, A K-major, B N-major, D row."""
    path = _run_case(oracle, 256, 128, 512, "bias", "k", "n", "row", dist=("uniform01", 1.0))
    assert path == ge.GE_PATH_TC_GEMM


@pytest.mark.parametrize("epi", ["bias", "relu_bias", "gelu_bias"])
def test_config2(oracle, epi):
    """1024x512x2048, N(0,1)/sqrt(2048) operands, N(0,1) bias."""
    _run_case(oracle, 1024, 512, 2048, epi, "k", "n", "row", dist=("normal", 2048 ** -0.5), seed=1)


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (129, 17, 128)])
@pytest.mark.parametrize("epi", ["none", "bias", "relu_bias", "relu_aux_bias"])
@pytest.mark.parametrize("am,bm,dl", [("k", "n", "row"), ("k", "k", "col"), ("m", "n", "row"),
                                      ("m", "k", "col")])
def test_exact_integer(oracle, M, N, K, epi, am, bm, dl):
    """Integer data: every partial sum is exact in fp32 and fp16, so the GPU
    must reproduce the oracle bit for bit (values and mask)."""
    _run_case(oracle, M, N, K, epi, am, bm, dl, dist=("int", 2.0), seed=2, exact=True)


SHAPES = [(1, 1, 1), (7, 33, 9), (128, 256, 64), (129, 257, 65), (300, 520, 200), (64, 1000, 136),
          (520, 40, 1032), (257, 129, 4100)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("am,bm,dl", list(itertools.product("km", "kn", ("row", "col"))))
def test_layouts_ragged(oracle, M, N, K, am, bm, dl):
    epi = EPIS[(M + N + K + len(am + bm + dl)) % len(EPIS)]
    _run_case(oracle, M, N, K, epi, am, bm, dl, seed=3)


@pytest.mark.parametrize("producers", ["0", "1"])
@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("am,bm", [("k", "k"), ("m", "n"), ("k", "n"), ("m", "k")])
def test_one_or_two_producer_warps(oracle, monkeypatch, producers, pair, am, bm):
    """The B loads issued by the stage's producer or by a second producer
    warp on the same barriers (by default only when an operand is M/N-major),
    forced both ways on every operand major, single-CTA and pair tiles,
    ragged edges; bit-exact on integer data."""
    monkeypatch.setenv("GE_TWO_PRODUCERS", producers)
    monkeypatch.setenv("GE_PAIR", pair)
    monkeypatch.setenv("GE_TILE_N", "256" if pair == "1" else "128")
    _run_case(oracle, 1000, 1160, 1032, "relu_aux_bias", am, bm, "row", dist=("int", 1.0), seed=24, exact=True)


@pytest.mark.parametrize("epi", EPIS)
def test_every_epilogue_multi_tile(oracle, epi):
    """Several tiles in both directions, ragged tails, K not a multiple of 64."""
    _run_case(oracle, 700, 900, 328, epi, "k", "n", "row", seed=4)
    _run_case(oracle, 700, 900, 328, epi, "k", "k", "col", seed=5)


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8, 13, 16])
@pytest.mark.parametrize("epi", ["none", "bias", "relu_bias", "gelu_bias"])
def test_few_token_paths(oracle, N, epi):
    """Up to 4 tokens the weight-streaming GEMV, from 5 the tensor-core
    kernel (D's stride a multiple of 8)."""
    want = ge.GE_PATH_GEMV if N <= 4 else ge.GE_PATH_TC_GEMM
    path = _run_case(oracle, 1000, N, 1000, epi, "k", "k", "col", seed=6)
    assert path == want
    path = _run_case(oracle, 333, N, 4104, epi, "k", "k", "row", seed=7)
    assert path == want


@pytest.mark.parametrize("N", [5, 7, 13, 15])
def test_gemv_few_tokens_unaligned_d(oracle, N):
    """5 to 16 tokens with D row-major and a stride of N (not a multiple of
    8): the tensor-core kernel's stores need 16-byte rows, so the GEMV
    takes them."""
    M, K = 300, 520
    A = f16_tensor((M, K), 300 + N).cuda()
    B = f16_tensor((N, K), 310 + N).cuda()
    bias = f16_tensor((M,), 320 + N).cuda()
    D = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    L = ge.make_layout(ge.GE_K_MAJOR, ge.GE_K_MAJOR, ge.GE_D_ROW, ldd=N)
    with ge.Plan(M, N, K, ge.GE_EPI_GELU_BIAS, L) as p:
        assert p.path == ge.GE_PATH_GEMV
        p.execute(A, B, bias, D)
        torch.cuda.synchronize()
    ref = oracle.linear_forward(bits(A), bits(B), bits(bias), "gelu_bias", M, N, K,
                                a_major="k", b_major="k", d_layout="row")
    check_f16(oracle, bits(D).reshape(-1), ref["D"], f"gemv {M}x{N}x{K} ldd {N}")


@pytest.mark.parametrize("N,dl", [(1, "col"), (3, "col"), (8, "col"), (16, "col"), (5, "row"), (16, "row")])
def test_mask_epilogue_with_few_tokens(oracle, N, dl):
    """RELU_AUX_BIAS with a handful of tokens takes the tensor-core path (the
    GEMV has no mask output): its 128-wide tiles hold 1 to 16 valid rows (D
    column-major, operands swapped; the one wave of tiles is then split
    along K) or columns (D row-major)."""
    path = _run_case(oracle, 1000, N, 1000, "relu_aux_bias", "k", "k", dl, seed=90 + N)
    assert path == ge.GE_PATH_TC_GEMM


@pytest.mark.parametrize("epi", ["bias", "relu_bias", "gelu_bias", "relu_aux_bias"])
def test_unfused_baseline(oracle, epi):
    """The three-kernel baseline computes the same values (its mask comes from
    the rounded fp16 z, which only differs inside the tolerance band)."""
    _run_case(oracle, 520, 264, 200, epi, "k", "n", "row", seed=8, unfused=True)
    _run_case(oracle, 520, 264, 200, epi, "k", "k", "col", seed=9, unfused=True)
    _run_case(oracle, 301, 90, 64, epi, "k", "k", "col", seed=10, unfused=True)   # rows end 5 short of 8
    _run_case(oracle, 96, 263, 64, epi, "m", "n", "row", seed=11, unfused=True)   # rows end 7 short of 8


def test_repeat_is_deterministic():
    A = f16_tensor((512, 512), 11).cuda()
    B = f16_tensor((512, 512), 12).cuda()
    bias = f16_tensor((512,), 13).cuda()
    w = Workload("det", 512, 512, 512, "gelu_bias", "k", "n", "row")
    d1, _, _, _ = gpu_forward(w, A, B, bias)
    d2, _, _, _ = gpu_forward(w, A, B, bias)
    assert torch.equal(d1.view(torch.int16), d2.view(torch.int16))


def test_timeout_probe_reports_and_recovers():
    """A bounded wait that nothing satisfies expires, is reported once, and
    leaves the context usable."""
    with ge.Plan(128, 128, 64, ge.GE_EPI_BIAS) as p:
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
        assert ge.ge_debug_wait_timeout(p.handle, 2_000_000) == ge.GE_OK
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_ERR_TIMEOUT
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK  # read clears it
        A = torch.ones(128, 64, dtype=torch.float16, device="cuda")
        B = torch.ones(64, 128, dtype=torch.float16, device="cuda")
        bias = torch.zeros(128, dtype=torch.float16, device="cuda")
        D = torch.empty(128, 128, dtype=torch.float16, device="cuda")
        p.execute(A, B, bias, D)
        torch.cuda.synchronize()
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
        assert torch.all(D == 64)


def test_execute_rejects_bad_buffers():
    with ge.Plan(128, 128, 64, ge.GE_EPI_RELU_AUX_BIAS) as p:
        A = torch.ones(128, 64, dtype=torch.float16, device="cuda")
        B = torch.ones(64, 128, dtype=torch.float16, device="cuda")
        bias = torch.zeros(128, dtype=torch.float16, device="cuda")
        D = torch.empty(128, 128, dtype=torch.float16, device="cuda")
        aux = torch.empty(p.aux_bytes // 4, dtype=torch.int32, device="cuda")
        assert ge.ge_execute(p.handle, A, B, bias, D, None, raw=True) == ge.GE_ERR_INVALID_ARG
        assert ge.ge_execute(p.handle, A, B, None, D, aux, raw=True) == ge.GE_ERR_INVALID_ARG
        assert ge.ge_execute(p.handle, A.data_ptr() + 2, B, bias, D, aux, raw=True) == ge.GE_ERR_ALIGNMENT
        host = torch.ones(128, 64, dtype=torch.float16)
        assert ge.ge_execute(p.handle, host, B, bias, D, aux, raw=True) == ge.GE_ERR_DEVICE_MISMATCH
        assert ge.ge_execute(p.handle, A, B, bias, D, aux, raw=True) == ge.GE_OK
        torch.cuda.synchronize()


PAIR_SHAPES = [(300, 520, 200), (257, 129, 4100), (700, 900, 328), (1000, 2056, 96), (513, 264, 64)]


@pytest.mark.parametrize("M,N,K", PAIR_SHAPES)
@pytest.mark.parametrize("am,bm,dl", [("k", "n", "row"), ("k", "k", "col"), ("m", "n", "row"),
                                      ("m", "k", "col")])
def test_pair_tiles_ragged(oracle, monkeypatch, M, N, K, am, bm, dl):
    """2-CTA (256-row) tiles forced on: ragged edges, every operand major."""
    monkeypatch.setenv("GE_PAIR", "1")
    monkeypatch.setenv("GE_TILE_N", "256")
    epi = EPIS[(M + N + K) % len(EPIS)]
    _run_case(oracle, M, N, K, epi, am, bm, dl, seed=20)


@pytest.mark.parametrize("epi", ["none", "bias", "relu_aux_bias"])
def test_pair_tiles_exact_integer(oracle, monkeypatch, epi):
    monkeypatch.setenv("GE_PAIR", "1")
    monkeypatch.setenv("GE_TILE_N", "256")
    _run_case(oracle, 520, 776, 128, epi, "k", "n", "row", dist=("int", 2.0), seed=21, exact=True)
    _run_case(oracle, 520, 776, 128, epi, "m", "k", "col", dist=("int", 2.0), seed=22, exact=True)


@pytest.mark.parametrize("am,bm,dl", [("k", "n", "row"), ("k", "k", "col"), ("m", "n", "row"),
                                      ("m", "k", "col")])
def test_pair_tiles_128_wide(oracle, monkeypatch, am, bm, dl):
    """2-CTA pairs of 256 x 128 tiles (each CTA stages 64 columns of B):
    K a multiple of 128 (two panels a stage) and a ragged K (one)."""
    monkeypatch.setenv("GE_PAIR", "1")
    monkeypatch.setenv("GE_TILE_N", "128")
    for M, N, K, seed in ((520, 776, 1024, 40), (300, 264, 520, 41)):
        _run_case(oracle, M, N, K, EPIS[seed % len(EPIS)], am, bm, dl, seed=seed)


@pytest.mark.parametrize("kb", ["64", "128"])
@pytest.mark.parametrize("epi", ["none", "relu_aux_bias"])
def test_stage_panels_exact_integer(oracle, monkeypatch, kb, epi):
    """One or two 64-wide k panels per pipeline stage (GE_KB) on a K that is
    a multiple of 128, single-CTA and pair tiles, integer data: bit-identical
    to the oracle either way."""
    monkeypatch.setenv("GE_KB", kb)
    for pair in ("0", "1"):
        monkeypatch.setenv("GE_PAIR", pair)
        _run_case(oracle, 520, 776, 384, epi, "k", "n", "row", dist=("int", 2.0), seed=42, exact=True)
        _run_case(oracle, 520, 776, 384, epi, "m", "k", "col", dist=("int", 2.0), seed=43, exact=True)


@pytest.mark.parametrize("epi", EPIS + ["gelu_erf_bias"])
def test_pair_tiles_224_wide(oracle, monkeypatch, epi):
    """256 x 224 pair tiles (112 B' rows a CTA, 448 of 512 TMEM columns):
    K-major B' only; N a multiple of 224, ragged (a last tile 64 wide, and
    odd), integer data bit-identical, normal data in tolerance."""
    monkeypatch.setenv("GE_TILE_N", "224")
    monkeypatch.setenv("GE_PAIR", "1")
    L = ge.make_layout(ge.GE_K_MAJOR, ge.GE_K_MAJOR, ge.GE_D_COL)
    with ge.Plan(1344, 512, 512, ge.EPILOGUE_BY_NAME[epi], L) as p:
        assert p.config[1:4] == (224, 1, 1)
    exact = epi not in ("gelu_bias", "gelu_erf_bias")
    dist = ("int", 2.0) if exact else ("normal", 1.0)
    # D column-major: the kernel's N is M (1344 = 6 x 224; 1000; 4096 = 18 x 224 + 64)
    _run_case(oracle, 1344, 512, 512, epi, "k", "k", "col", dist=dist, seed=80, exact=exact)
    _run_case(oracle, 1000, 300, 640, epi, "k", "k", "col", dist=dist, seed=81, exact=exact)
    _run_case(oracle, 520, 776, 384, epi, "m", "k", "row", dist=dist, seed=82, exact=exact)


def test_pair_tiles_224_chosen_for_two_ragged_waves():
    """The planner takes 256 x 224 pair tiles where 256 x 256 ones leave a
    second wave too full for the split tail (FFN up-projection, T = 2048),
    and never for an N-major B'."""
    L = ge.make_layout(ge.GE_K_MAJOR, ge.GE_K_MAJOR, ge.GE_D_COL)
    with ge.Plan(4096, 2048, 4096, ge.GE_EPI_GELU_BIAS, L) as p:
        assert p.config[1:4] == (224, 1, 1), p.config
    Ln = ge.make_layout(ge.GE_K_MAJOR, ge.GE_MN_MAJOR, ge.GE_D_ROW)
    with ge.Plan(2048, 4096, 4096, ge.GE_EPI_GELU_BIAS, Ln) as p:
        assert p.config[1] != 224, p.config


@pytest.mark.parametrize("epi", ["none", "bias", "relu_aux_bias"])
def test_split_tail_exact_integer(oracle, epi):
    """Split-K tail (4 tiles split 4 ways, then the fixup kernel): integer
    data keeps every partial sum exact, so the result is still bit-identical."""
    _run_case(oracle, 256, 256, 1024, epi, "k", "n", "row", dist=("int", 1.0), seed=30, exact=True)
    _run_case(oracle, 256, 256, 1024, epi, "m", "k", "col", dist=("int", 1.0), seed=31, exact=True)


@pytest.mark.parametrize("epi", EPIS)
def test_split_tail_pair_ragged(oracle, monkeypatch, epi):
    """Pair tiles with a split-K tail on ragged extents."""
    monkeypatch.setenv("GE_PAIR", "1")
    monkeypatch.setenv("GE_TILE_N", "256")
    _run_case(oracle, 1000, 2056, 520, epi, "k", "n", "row", seed=32)
    _run_case(oracle, 1000, 2056, 520, epi, "k", "k", "col", seed=33)


@pytest.mark.parametrize("epi", ["bias", "relu_aux_bias", "gelu_bias"])
def test_underfilled_problem_split_whole(oracle, epi):
    """A single wave that leaves most SMs idle (config 2: 32 tiles of 128 x 128)
    is split along K as a whole, 4 pieces per tile, and the fixup applies the
    epilogue: bit-identical on integer data, within tolerance otherwise."""
    L = ge.make_layout(ge.GE_K_MAJOR, ge.GE_MN_MAJOR, ge.GE_D_ROW)
    with ge.Plan(1024, 512, 2048, ge.EPILOGUE_BY_NAME[epi], L) as p:
        path, bn, pair, split = p.config
        assert (path, bn, pair, split) == (ge.GE_PATH_TC_GEMM, 128, 0, 4)
    if epi != "gelu_bias":
        _run_case(oracle, 1024, 512, 2048, epi, "k", "n", "row", dist=("int", 1.0), seed=35, exact=True)
    _run_case(oracle, 1024, 512, 2048, epi, "k", "n", "row", seed=36)


def test_split_tail_matches_unsplit(oracle, monkeypatch):
    """The same problem with and without the split tail agrees with the oracle."""
    for flag in ("0", "1"):
        monkeypatch.setenv("GE_SPLIT_TAIL", flag)
        _run_case(oracle, 300, 520, 1024, "gelu_bias", "k", "n", "row", seed=34)


@pytest.mark.parametrize("M,N,K", [(4096, 1, 8192), (4096, 3, 8192), (2000, 2, 1024), (1500, 4, 4096)])
def test_gemv_many_rows_per_warp(oracle, M, N, K):
    """GEMV shapes with more rows than warps of the grid, K up to 8192."""
    path = _run_case(oracle, M, N, K, "gelu_bias", "k", "k", "col", seed=60 + N)
    assert path == ge.GE_PATH_GEMV


@pytest.mark.parametrize("M,K", [(4096, 4096), (12000, 4096), (1000, 4104), (700, 1000)])
def test_gemv_static_weights_preload(oracle, M, K):
    """One token with static weights: the first slabs of each warp's first row
    are loaded before the wait on the previous grid; rows beyond the grid's
    warps (12000), a ragged K (4104) and rows shorter than the preload (1000)."""
    L = ge.make_layout(ge.GE_K_MAJOR, ge.GE_K_MAJOR, ge.GE_D_COL)
    W = f16_tensor((M, K), 730 + M, "normal", K ** -0.5).cuda()
    x = f16_tensor((1, K), 731).cuda()
    b = f16_tensor((M,), 732, "normal", 0.1).cuda()
    with ge.Plan(M, 1, K, ge.GE_EPI_GELU_BIAS, L) as p:
        p.set_attr(ge.GE_ATTR_STATIC_A, 1)
        assert p.path == ge.GE_PATH_GEMV
        y = torch.full((1, M), float("nan"), dtype=torch.float16, device="cuda")
        p.execute(W, x, b, y)
        p.execute(W, x, b, y)  # a second launch depends on the first
        torch.cuda.synchronize()
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
    r = oracle.linear_forward(bits(W), bits(x), bits(b), "gelu_bias", M, 1, K, a_major="k", b_major="k",
                              d_layout="col")
    check_f16(oracle, bits(y), r["D"], f"static gemv {M}x1x{K}")


def test_gemv_chain_with_static_weights(oracle):
    """A chain of decode projections (each layer's output is the next one's
    input, ping-pong buffers) launched with programmatic dependent launch:
    every layer still waits for its input and for the previous reader of its
    output buffer. Checked layer by layer against the oracle's own chain."""
    H, layers = 2048, 4
    Ws = [f16_tensor((H, H), 700 + i, "normal", H ** -0.5).cuda() for i in range(layers)]
    bs = [f16_tensor((H,), 710 + i, "normal", 0.1).cuda() for i in range(layers)]
    x0 = f16_tensor((1, H), 720).cuda()
    bufs = [x0.clone(), torch.empty_like(x0)]
    L = ge.make_layout(ge.GE_K_MAJOR, ge.GE_K_MAJOR, ge.GE_D_COL)
    plans = [ge.Plan(H, 1, H, ge.GE_EPI_GELU_BIAS, L) for _ in range(layers)]
    for p in plans:
        p.set_attr(ge.GE_ATTR_STATIC_A, 1)
        assert p.path == ge.GE_PATH_GEMV
    for i, p in enumerate(plans):
        src, dst = bufs[i % 2], bufs[(i + 1) % 2]  # layer i+1 overwrites layer i's input
        p.execute(Ws[i], src, bs[i], dst)
    torch.cuda.synchronize()
    for p in plans:
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
        p.free()
    # the same chain with a fresh buffer per layer, to compare every stage
    got = []
    cur = x0.clone()
    plans = [ge.Plan(H, 1, H, ge.GE_EPI_GELU_BIAS, L) for _ in range(layers)]
    for i, p in enumerate(plans):
        p.set_attr(ge.GE_ATTR_STATIC_A, 1)
        nxt = torch.empty_like(x0)
        p.execute(Ws[i], cur, bs[i], nxt)
        got.append(nxt)
        cur = nxt
    torch.cuda.synchronize()
    # the ping-pong chain's final output equals the step-by-step one
    assert torch.equal(bufs[layers % 2], got[-1])
    ref_in = bits(x0)
    for i in range(layers):
        r = oracle.linear_forward(bits(Ws[i]), ref_in, bits(bs[i]), "gelu_bias", H, 1, H,
                                  a_major="k", b_major="k", d_layout="col")
        check_f16(oracle, bits(got[i]), r["D"], f"chain layer {i}")
        ref_in = r["D"]
    for p in plans:
        p.free()


@pytest.mark.parametrize("am,bm,dl", [("k", "n", "row"), ("k", "k", "col"), ("m", "n", "row"), ("m", "k", "col")])
def test_gelu_erf_epilogue(oracle, am, bm, dl):
    """Exact (erf) GELU: single-CTA tiles, ragged edges, every operand major."""
    _run_case(oracle, 300, 520, 200, "gelu_erf_bias", am, bm, dl, seed=80)


def test_gelu_erf_pair_gemv_unfused(oracle, monkeypatch):
    _run_case(oracle, 1000, 3, 1000, "gelu_erf_bias", "k", "k", "col", seed=81)      # GEMV
    _run_case(oracle, 520, 264, 200, "gelu_erf_bias", "k", "n", "row", seed=82, unfused=True)
    monkeypatch.setenv("GE_PAIR", "1")
    monkeypatch.setenv("GE_TILE_N", "256")
    _run_case(oracle, 1000, 2056, 520, "gelu_erf_bias", "k", "k", "col", seed=83)  # pairs + split tail


def test_autotune_picks_a_candidate_and_stays_correct(oracle):
    """Plan-time selection by timing: the chosen configuration is one of the
    candidates, the outputs it leaves are correct, and later executes agree."""
    M, N, K = 1500, 2056, 1024
    w = Workload("autotune", M, N, K, "relu_aux_bias", "k", "n", "row")
    A, B, bias = w.make("cuda")
    with ge.Plan(M, N, K, ge.GE_EPI_RELU_AUX_BIAS, ge.make_layout(ge.GE_K_MAJOR, ge.GE_MN_MAJOR, ge.GE_D_ROW)) as p:
        D = torch.empty((M, N), dtype=torch.float16, device="cuda")
        aux = torch.empty(p.aux_bytes // 4, dtype=torch.int32, device="cuda")
        p.autotune(A, B, bias, D, aux, reps=3)
        torch.cuda.synchronize()
        path, bn, pair, split = p.config
        assert path == ge.GE_PATH_TC_GEMM and bn in (128, 256) and pair in (0, 1, 2) and split >= 1
        assert not (pair and bn != 256)
        ref = oracle_full(oracle, w, A.cpu(), B.cpu(), bias.cpu())
        check_f16(oracle, bits(D), ref["D"], "autotuned")
        check_mask(aux.cpu().numpy().view(np.uint32), ref["aux"], ref["Z"], M, N, p.aux_ld, "autotuned")
        D2 = torch.empty_like(D)
        p.execute(A, B, bias, D2, aux)
        torch.cuda.synchronize()
        assert torch.equal(D.view(torch.int16), D2.view(torch.int16))
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
        tuned = p.config
    # a later plan for the same problem starts from the tuned configuration
    L = ge.make_layout(ge.GE_K_MAJOR, ge.GE_MN_MAJOR, ge.GE_D_ROW)
    with ge.Plan(M, N, K, ge.GE_EPI_RELU_AUX_BIAS, L) as p2:
        assert p2.config == tuned
    ge.ge_autotune_cache_clear()
    with ge.Plan(M, N, K, ge.GE_EPI_RELU_AUX_BIAS, L) as p3:
        assert p3.config[0] == ge.GE_PATH_TC_GEMM


def test_autotune_k_major_candidates_stay_correct(oracle):
    """With a K-major B' the candidates also hold 224-wide pair tiles and
    stages of one or two k panels; whichever wins, the outputs it leaves
    match the oracle and a later plan for the problem starts from it."""
    M, N, K = 1344, 600, 1024
    w = Workload("autotune k-major", M, N, K, "gelu_bias", "k", "k", "col")
    A, B, bias = w.make("cuda")
    L = ge.make_layout(ge.GE_K_MAJOR, ge.GE_K_MAJOR, ge.GE_D_COL)
    with ge.Plan(M, N, K, ge.GE_EPI_GELU_BIAS, L) as p:
        D = torch.empty(w.d_shape(), dtype=torch.float16, device="cuda")
        p.autotune(A, B, bias, D, None, reps=2)
        torch.cuda.synchronize()
        path, bn, pair, split = p.config
        assert path == ge.GE_PATH_TC_GEMM and bn in (128, 224, 256)
        assert not (bn == 224 and (not pair or split != 1))
        ref = oracle_full(oracle, w, A.cpu(), B.cpu(), bias.cpu())
        check_f16(oracle, bits(D), ref["D"], "autotuned k-major")
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
        tuned = p.config
    with ge.Plan(M, N, K, ge.GE_EPI_GELU_BIAS, L) as p2:
        assert p2.config == tuned
    ge.ge_autotune_cache_clear()


@pytest.mark.parametrize("epi", EPIS + ["gelu_erf_bias"])
@pytest.mark.parametrize("kind", ["zeros", "overflow", "nan"])
def test_degenerate_values(oracle, epi, kind):
    """Zero operands (D = act(bias)), results beyond fp16 range (rounded to
    +-inf on both sides) and NaN inputs (propagated by the product; ReLU maps
    NaN to 0 on both sides, the mask bit of NaN is 0)."""
    M, N, K = 160, 96, 64
    w = Workload(f"{kind} {epi}", M, N, K, epi, "k", "n", "row")
    A = f16_tensor((M, K), 90, "normal", 1.0)
    B = f16_tensor((K, N), 91, "normal", 1.0)
    bias = f16_tensor((M,), 92, "normal", 1.0)
    if kind == "zeros":
        A.zero_()
    elif kind == "overflow":
        A[:8] = 200.0           # 64 * 200 * |B| exceeds 65504 for many entries
        B[:, :8] = 250.0
    else:
        A[3, 5] = float("nan")  # row 3 of D is NaN (before the activation)
        B[7, 11] = float("nan")  # column 11 of D is NaN
    A, B, bias = A.cuda(), B.cuda(), bias.cuda()
    D, aux, path, ld_aux = gpu_forward(w, A, B, bias)
    ref = oracle_full(oracle, w, A.cpu(), B.cpu(), bias.cpu())
    got = oracle.f16_decode(bits(D))
    want = oracle.f16_decode(ref["D"])
    assert np.array_equal(np.isnan(got), np.isnan(want)), "NaN positions differ"
    assert np.array_equal(np.isinf(got), np.isinf(want)), "inf positions differ"
    fin = np.isfinite(want)
    assert np.array_equal(np.sign(got[~fin & ~np.isnan(want)]), np.sign(want[~fin & ~np.isnan(want)]))
    err = np.abs(got[fin] - want[fin])
    assert (err <= 1e-2 * np.maximum(1.0, np.abs(want[fin]))).all()
    if epi == "relu_aux_bias":
        z = ref["Z"].reshape(M, N)
        sure = np.abs(np.nan_to_num(z, nan=1.0)) > 1e-3
        from _util import mask_bits
        g = mask_bits(aux.cpu().numpy().view(np.uint32), M, ld_aux, N)
        r = mask_bits(ref["aux"], M, ld_aux, N)
        assert np.array_equal(g[sure], r[sure])
