"""Host-side logic of the benchmark (no GPU): which measured peak a timing is
held to, the percentile helper, and the oracle baselines of the config table
on tiny problems in both of their forms (whole problem, sampled rows)."""
import math
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from gemm_epilogues_gb300.inputs import Workload, f16_tensor  # noqa: E402

PEAKS = {"tflops": 1900.0, "tflops_sustained": 1700.0, "hbm_gbs": 6700.0}


def test_short_region_uses_burst_even_when_capped():
    peak, sustained, capped = bench.choose_tensor_peak(PEAKS, 0.02, {"reasons": ["sw_power_cap"]})
    assert (peak, sustained, capped) == (1900.0, False, True)


def test_long_capped_region_uses_sustained():
    peak, sustained, _ = bench.choose_tensor_peak(PEAKS, 2.5, {"reasons": ["sw_power_cap"]})
    assert (peak, sustained) == (1700.0, True)


def test_long_region_without_cap_uses_burst():
    assert bench.choose_tensor_peak(PEAKS, 2.5, {"reasons": []})[0] == 1900.0
    assert bench.choose_tensor_peak(PEAKS, 2.5, None)[0] == 1900.0


def test_percentile():
    xs = list(range(1, 51))  # 1..50
    assert bench._pct(xs, 0.9) == 45
    assert bench._pct(xs, 0.5) == 25
    assert bench._pct([3.0], 0.9) == 3.0


def test_oracle_config_baselines_whole_and_sampled():
    w = Workload("tiny", 24, 16, 32, "relu_aux_bias", "k", "k", "col")
    A = f16_tensor((24, 32), 11)
    B = f16_tensor((16, 32), 12)
    b = f16_tensor((24,), 13)
    cpu_in = {"cfg_c3_T512": ("full", A, B, b, w, None),
              "cfg_c4_fwd": ("sample", A, B[:4], b, w, 16)}
    out = bench.oracle_config_baselines(cpu_in)
    full, samp = out["cfg_c3_T512"], out["cfg_c4_fwd"]
    assert full["sample"] == "whole problem" and full["tflops"] > 0
    assert samp["sample"] == "4 of 16 stored rows of D"
    # the sampled time is scaled to the whole problem by the ratio of rows
    assert math.isclose(samp["extrapolated_s"], samp["s"] * 16 / 4)


def test_oracle_config_baselines_drelu():
    M, N = 40, 8
    ld_aux = (M + 127) // 128 * 4
    dY = f16_tensor((N, M), 21)
    aux = torch.randint(-2**31, 2**31 - 1, (N * ld_aux,), dtype=torch.int32,
                        generator=torch.Generator().manual_seed(22))
    out = bench.oracle_config_baselines({"cfg_c4_bwd": (dY, aux, M, N, ld_aux)})
    assert out["cfg_c4_bwd"]["gbs"] > 0 and out["cfg_c4_bwd"]["sample"] == "whole problem"
