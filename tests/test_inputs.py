"""The seeded input generators and the workload bookkeeping, on the CPU:
determinism, the value ranges the recipe promises, the sampled-row sets, and
the per-workload flop and byte counts against the figures worked out by hand
from the shapes (operands read once, D written once, bias read, one mask bit
per element of D in rows padded to 128 bits)."""
import numpy as np
import pytest
import torch

from gemm_epilogues_gb300.inputs import f16_tensor, pages_workloads, sample_rows


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_uniform_draws_stay_below_one(dtype):
    x = f16_tensor((1 << 16,), 7, dist="uniform01", dtype=dtype).float()
    assert (x >= 0).all() and (x < 1).all()
    assert x.max() > 0.99  # the clamp keeps values, it does not shrink the range


def test_same_seed_same_draws_for_either_type():
    a = f16_tensor((257, 33), 11)
    b = f16_tensor((257, 33), 11)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    h = f16_tensor((257, 33), 11, dtype=torch.bfloat16).float()
    # both are one rounding of the same fp32 draw
    assert torch.allclose(a.float(), h, rtol=2 ** -7, atol=0)
    assert not torch.equal(a, f16_tensor((257, 33), 12))


def test_integer_draws_are_exact_and_in_range():
    x = f16_tensor((4096,), 5, dist="int", std=2).float()
    assert torch.equal(x, x.round())
    assert set(x.unique().tolist()) == {-2.0, -1.0, 0.0, 1.0, 2.0}


def test_normal_scale():
    x = f16_tensor((1 << 18,), 3, std=1 / 64).double()
    assert abs(x.std().item() * 64 - 1) < 0.01
    assert abs(x.mean().item()) < 1e-4


@pytest.mark.parametrize("n", [1, 255, 256, 257, 8192, 65536])
def test_sample_rows(n):
    r = sample_rows(n)
    assert len(r) == min(n, 256)
    assert len(np.unique(r)) == len(r) and (np.diff(r) > 0).all()
    assert r[0] >= 0 and r[-1] < n
    assert np.array_equal(r, sample_rows(n))
    if n > 256:
        assert not np.array_equal(r, sample_rows(n, seed=1))


def test_workload_counts():
    w = pages_workloads()
    # forward of the MLP layer: 2*(W + X + Y) + 2*bias + 8192 token rows x
    # 86 sixteen-byte mask chunks (11008 features = 86 x 128 bits)
    c4 = w["c4_fwd"]
    assert c4.flops == 2 * 11008 * 8192 * 4096 == 738_734_374_912
    assert c4.algorithmic_bytes() == 337_641_472 + 22_016 + 8192 * 86 * 16 == 348_935_680
    assert w["c4_dw"].algorithmic_bytes() == 337_641_472 + 22_016
    c5 = w["c5"]
    assert c5.flops == 17_592_186_044_416
    # row-major D [65536, 8192]: 64 mask chunks per row
    assert c5.algorithmic_bytes() == 2 * (65536 * 16384 + 16384 * 8192 + 65536 * 8192) + 2 * 65536 \
        + 65536 * 64 * 16
    d = w["c3_T1"]
    assert (d.M, d.N, d.K) == (4096, 1, 4096)
    assert d.algorithmic_bytes() == 2 * (4096 * 4096 + 4096 + 4096) + 2 * 4096
    assert w["c1"].a_shape() == (256, 512) and w["c1"].b_shape() == (512, 128)
    assert c4.a_shape() == (11008, 4096) and c4.b_shape() == (8192, 4096) and c4.d_shape() == (8192, 11008)
