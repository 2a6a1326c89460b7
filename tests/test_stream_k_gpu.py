"""Stream-K tiles of the tensor-core GEMM: the last waves' tiles are shared
out as equal ranges of k-block iterations, and a tile cut between workers is
finished inside the GEMM by the worker whose range starts it (it adds the
others' fp32 pieces in k order). Parity with the oracle element by element:
bit-identical on integer data (every partial sum is exact in fp32), within
tolerance otherwise; pair and single-CTA tiles, data-parallel waves before
the stream-K ones, workers with empty ranges, ragged extents, every forward
epilogue, bf16; repeated launches and CUDA-graph replays (the flags that
order the pieces carry a per-launch epoch)."""
import pytest
import torch

import gemm_epilogues_gb300 as ge
from gemm_epilogues_gb300.inputs import f16_tensor

from test_gemm_gpu import EPIS, _run_case

pytestmark = pytest.mark.gpu


def _force(monkeypatch, pair, tile_n):
    monkeypatch.setenv("GE_STREAM_K", "1")
    monkeypatch.setenv("GE_PAIR", pair)
    monkeypatch.setenv("GE_TILE_N", tile_n)


def _sk_tiles(M, N, K, epi="bias", am=ge.GE_K_MAJOR, bm=ge.GE_MN_MAJOR, dl=ge.GE_D_ROW):
    with ge.Plan(M, N, K, ge.EPILOGUE_BY_NAME[epi], ge.make_layout(am, bm, dl)) as p:
        return p.stream_k_tiles, p.config


def test_planner_takes_stream_k_only_when_asked(monkeypatch):
    # FFN up-projection T = 2048 in 256-wide pair tiles (left alone the
    # planner takes 224-wide ones there): 128 tiles on the pairs of SMs; by
    # default two plain waves, with GE_STREAM_K = 1 stream-K over all of them
    monkeypatch.setenv("GE_TILE_N", "256")
    n, cfg = _sk_tiles(4096, 2048, 4096, "gelu_bias", ge.GE_K_MAJOR, ge.GE_K_MAJOR, ge.GE_D_COL)
    assert n == 0 and cfg[3] == 1, (n, cfg)
    monkeypatch.setenv("GE_STREAM_K", "1")
    n, cfg = _sk_tiles(4096, 2048, 4096, "gelu_bias", ge.GE_K_MAJOR, ge.GE_K_MAJOR, ge.GE_D_COL)
    assert n > 0 and cfg[3] == 1, (n, cfg)
    # a problem that fills its waves exactly has nothing to share out
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n, _ = _sk_tiles(128 * sms, 128, 256)
    assert n == 0
    # backward epilogues never take it (their bias-gradient partials are per tile)
    n, _ = _sk_tiles(4096, 2048, 4096, "drelu_bgrad")
    assert n == 0
    monkeypatch.setenv("GE_STREAM_K", "0")
    n, cfg = _sk_tiles(11008, 8192, 4096, "relu_aux_bias", ge.GE_K_MAJOR, ge.GE_K_MAJOR, ge.GE_D_COL)
    assert n == 0 and cfg[3] > 1, (n, cfg)


@pytest.mark.parametrize("epi", ["none", "bias", "relu_aux_bias"])
def test_pair_tiles_exact_integer(oracle, monkeypatch, epi):
    """48 pair tiles of 256 x 256 over all pairs (K = 1024: 8 iterations a
    tile, ~5 a worker: every tile in 2-3 pieces)."""
    _force(monkeypatch, "1", "256")
    _run_case(oracle, 2048, 1536, 1024, epi, "k", "n", "row", dist=("int", 1.0), seed=60, exact=True)
    _run_case(oracle, 1536, 2048, 1024, epi, "m", "k", "col", dist=("int", 1.0), seed=61, exact=True)


@pytest.mark.parametrize("epi", ["bias", "relu_aux_bias"])
def test_single_cta_tiles_exact_integer(oracle, monkeypatch, epi):
    """96 tiles of 128 x 128 on single CTAs, 16 iterations of 64 k a tile."""
    _force(monkeypatch, "0", "128")
    monkeypatch.setenv("GE_KB", "64")
    _run_case(oracle, 1024, 1536, 1024, epi, "k", "n", "row", dist=("int", 1.0), seed=62, exact=True)
    monkeypatch.delenv("GE_KB")
    _run_case(oracle, 1024, 1536, 1024, epi, "k", "k", "col", dist=("int", 1.0), seed=63, exact=True)


def test_data_parallel_waves_then_stream_k_exact_integer(oracle, monkeypatch):
    """192 pair tiles: one data-parallel wave, then the last 116 tiles
    stream-K (a worker's whole tiles, its first piece spilled, its last
    finished)."""
    _force(monkeypatch, "1", "256")
    with ge.Plan(4096, 3072, 512, ge.GE_EPI_RELU_AUX_BIAS,
                 ge.make_layout(ge.GE_K_MAJOR, ge.GE_MN_MAJOR, ge.GE_D_ROW)) as p:
        assert 0 < p.stream_k_tiles < 192
    _run_case(oracle, 4096, 3072, 512, "relu_aux_bias", "k", "n", "row", dist=("int", 1.0), seed=64, exact=True)


@pytest.mark.parametrize("pair,tile_n,M,N,K", [("1", "256", 256, 256, 1024), ("0", "128", 128, 128, 2048),
                                                ("1", "256", 300, 200, 640)])
def test_more_workers_than_iterations_exact_integer(oracle, monkeypatch, pair, tile_n, M, N, K):
    """One tile and fewer k-block iterations than workers: most workers have
    an empty range, the finisher adds up to a dozen one-iteration pieces."""
    _force(monkeypatch, pair, tile_n)
    for epi in ("bias", "relu_aux_bias"):
        _run_case(oracle, M, N, K, epi, "k", "n", "row", dist=("int", 1.0), seed=65, exact=True)


@pytest.mark.parametrize("epi", EPIS + ["gelu_erf_bias"])
def test_ragged_every_epilogue(oracle, monkeypatch, epi):
    """Ragged rows, columns and K (520: stages of 64 k) with pair tiles."""
    _force(monkeypatch, "1", "256")
    _run_case(oracle, 1000, 2056, 520, epi, "k", "n", "row", seed=66)
    _run_case(oracle, 1000, 2056, 520, epi, "k", "k", "col", seed=67)


def test_bf16(oracle, monkeypatch):
    _force(monkeypatch, "1", "256")
    _run_case(oracle, 1000, 2056, 1024, "gelu_bias", "k", "n", "row", seed=68, dtype="bf16")
    _run_case(oracle, 1000, 2056, 1024, "relu_aux_bias", "m", "k", "col", dist=("int", 1.0), seed=69,
              exact=True, dtype="bf16")


def test_repeated_launches_and_graph_replays_are_identical(monkeypatch):
    """The same plan launched 40 times, then captured in a CUDA graph (three
    executes) and replayed: every output bit-identical to the first launch's
    (a stale flag from an earlier launch would let a finisher add a piece
    before it is written)."""
    _force(monkeypatch, "1", "256")
    M, N, K = 2048, 1536, 2048
    A = f16_tensor((M, K), 70).cuda()
    B = f16_tensor((K, N), 71).cuda()
    bias = f16_tensor((M,), 72).cuda()
    L = ge.make_layout(ge.GE_K_MAJOR, ge.GE_MN_MAJOR, ge.GE_D_ROW)
    with ge.Plan(M, N, K, ge.GE_EPI_GELU_BIAS, L) as p:
        assert p.stream_k_tiles > 0
        D0 = torch.empty((M, N), dtype=torch.float16, device="cuda")
        p.execute(A, B, bias, D0)
        torch.cuda.synchronize()
        D = torch.empty_like(D0)
        for _ in range(40):
            D.fill_(float("nan"))
            p.execute(A, B, bias, D)
        torch.cuda.synchronize()
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK
        assert torch.equal(D.view(torch.int16), D0.view(torch.int16))
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        outs = [torch.empty_like(D0) for _ in range(3)]
        with torch.cuda.stream(s):
            p.execute(A, B, bias, outs[0], None, s)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for o in outs:
                p.execute(A, B, bias, o, None, torch.cuda.current_stream())
        for _ in range(3):
            for o in outs:
                o.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            for o in outs:
                assert torch.equal(o.view(torch.int16), D0.view(torch.int16))
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK


def test_stream_k_and_split_tail_agree_with_the_oracle(oracle, monkeypatch):
    """The same ragged problem with stream-K off (split tail / whole split)
    and forced on."""
    monkeypatch.setenv("GE_PAIR", "1")
    monkeypatch.setenv("GE_TILE_N", "256")
    for flag in ("0", "1"):
        monkeypatch.setenv("GE_STREAM_K", flag)
        _run_case(oracle, 1300, 1800, 1536, "relu_aux_bias", "k", "n", "row", seed=73)
