"""The C ABI without a GPU: the library loads, exports every function the
header declares, and rejects invalid plans before touching the device."""
import os
import re

import pytest

import gemm_epilogues_gb300 as ge

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ge.h")


@pytest.fixture(scope="module")
def lib():
    from gemm_epilogues_gb300 import build
    build.build()
    return ge.load_library()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ge_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert header_functions() == sorted(ge.ABI_FUNCTIONS)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    for s in range(9):
        assert ge.ge_status_string(s).startswith("GE_")
    assert ge.ge_status_string(99) == "unknown ge_status_t"
    assert re.match(r"\d+\.\d+\.\d+", ge.ge_version())


def _create(*args, **kw):
    st, h = ge.ge_plan_create(*args, raw=True, **kw)
    assert h is None or st == ge.GE_OK
    return st


def test_plan_validation_without_device(lib):
    E = ge
    assert _create(0, 8, 8) == E.GE_ERR_INVALID_ARG
    assert _create(8, -1, 8) == E.GE_ERR_INVALID_ARG
    # empty problems are rejected on every path before the device is touched
    assert _create(8, 0, 8) == E.GE_ERR_INVALID_ARG
    assert _create(8, 0, 8, epi=E.GE_EPI_RELU_AUX_BIAS) == E.GE_ERR_INVALID_ARG
    assert _create(0, 8, 0, epi=E.GE_EPI_DRELU_BGRAD) == E.GE_ERR_INVALID_ARG
    assert _create(8, 0, 0, epi=E.GE_EPI_DRELU_BGRAD) == E.GE_ERR_INVALID_ARG
    assert _create(8, 0, 0, epi=E.GE_EPI_DGELU_BGRAD) == E.GE_ERR_INVALID_ARG
    assert _create(8, 8, 0, epi=E.GE_EPI_DW_DRELU_BGRAD,
                   layout=ge.make_layout(E.GE_MN_MAJOR, E.GE_MN_MAJOR, E.GE_D_ROW)) == E.GE_ERR_INVALID_ARG
    assert _create(8, 8, 0, epi=E.GE_EPI_BIAS) == E.GE_ERR_INVALID_ARG
    assert _create(8, 8, 8, epi=12) == E.GE_ERR_INVALID_ARG
    # the masked-operand weight gradient needs A read M-major and D row-major
    assert _create(8, 8, 8, epi=E.GE_EPI_DW_DRELU_BGRAD,
                   layout=ge.make_layout(E.GE_K_MAJOR, E.GE_MN_MAJOR, E.GE_D_ROW)) == E.GE_ERR_UNSUPPORTED
    assert _create(8, 8, 8, epi=E.GE_EPI_DW_DRELU_BGRAD,
                   layout=ge.make_layout(E.GE_MN_MAJOR, E.GE_MN_MAJOR, E.GE_D_COL)) == E.GE_ERR_UNSUPPORTED
    assert _create(64, 64, 64, epi=E.GE_EPI_DW_DRELU_BGRAD,
                   layout=ge.make_layout(E.GE_MN_MAJOR, E.GE_MN_MAJOR, E.GE_D_ROW, ld_aux=6)) == E.GE_ERR_ALIGNMENT
    # the norm epilogues need the features contiguous (D column-major)
    assert _create(8, 8, 8, epi=E.GE_EPI_BIAS_RESIDUAL_RMSNORM) == E.GE_ERR_UNSUPPORTED
    assert _create(8, 8, 8, a=E.GE_F32) == E.GE_ERR_UNSUPPORTED
    assert _create(8, 8, 8, compute=E.GE_F16) == E.GE_ERR_UNSUPPORTED
    # bf16 only when A, B and D are all bf16, and still with fp32 accumulation
    assert _create(8, 8, 8, a=E.GE_BF16) == E.GE_ERR_UNSUPPORTED
    assert _create(8, 8, 8, E.GE_BF16, E.GE_BF16, E.GE_F16) == E.GE_ERR_UNSUPPORTED
    assert _create(8, 8, 8, E.GE_BF16, E.GE_BF16, E.GE_BF16, E.GE_BF16) == E.GE_ERR_UNSUPPORTED
    assert _create(8, 8, 0, epi=E.GE_EPI_BIAS) == E.GE_ERR_INVALID_ARG
    assert _create(2**31, 8, 8) == E.GE_ERR_INVALID_ARG
    # leading dimensions smaller than the extent, or not multiples of 8
    assert _create(64, 64, 64, layout=ge.make_layout(lda=32)) == E.GE_ERR_INVALID_ARG
    assert _create(64, 60, 64, layout=ge.make_layout()) == E.GE_ERR_ALIGNMENT  # ldd = N = 60
    assert _create(64, 64, 60, layout=ge.make_layout(a=E.GE_K_MAJOR)) == E.GE_ERR_ALIGNMENT
    assert _create(64, 64, 0, epi=E.GE_EPI_DRELU_BGRAD,
                   layout=ge.make_layout(ld_aux=1)) == E.GE_ERR_INVALID_ARG
    assert _create(64, 300, 0, epi=E.GE_EPI_DRELU_BGRAD,
                   layout=ge.make_layout(ld_aux=10)) == E.GE_ERR_ALIGNMENT
    bad_layout = ge.make_layout()
    bad_layout.d = 7
    assert _create(64, 64, 64, layout=bad_layout) == E.GE_ERR_INVALID_ARG


def test_valid_plan_needs_a_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _create(256, 128, 512) == ge.GE_ERR_CUDA


def test_plan_attr_validation(lib):
    assert ge.ge_plan_set_attr(None, ge.GE_ATTR_STATIC_A, 1, raw=True) == ge.GE_ERR_INVALID_ARG
    assert ge.ge_plan_autotune(None, None, None, None, None, raw=True) == ge.GE_ERR_INVALID_ARG
    assert ge.ge_plan_config(None)[0] == -1
    assert ge.ge_plan_stream_k_tiles(None) == -1


def test_null_handles(lib):
    assert ge.load_library().ge_execute(None, None, None, None, None, None, None) == ge.GE_ERR_INVALID_ARG
    assert ge.load_library().ge_plan_free(None) == ge.GE_OK
    assert ge.ge_aux_bytes(None) == 0
    assert ge.ge_plan_path(None) == -1


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the built library every call raises: there is no fallback."""
    monkeypatch.setattr(ge, "_lib", None)
    monkeypatch.setattr(ge, "LIB_PATH", str(tmp_path / "libgemm_epilogues.so"))
    with pytest.raises(RuntimeError, match="not built"):
        ge.load_library()
    with pytest.raises(RuntimeError, match="not built"):
        ge.Plan(64, 64, 64, ge.GE_EPI_BIAS)
    with pytest.raises(RuntimeError, match="not built"):
        ge.ge_status_string(ge.GE_OK)
