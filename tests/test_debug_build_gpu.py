"""The checking build (GE_DEBUG): the same kernels compiled with device-side
checks of TMA coordinates and alignment, shared-memory stage and staging
offsets, TMEM column ranges, mask-word indices and the mbarrier phase
invariant (a producer never more than one phase of a stage ahead of its
consumer). A failed check records a bit in the plan's error word and skips
the access, so the context stays usable; ge_get_last_device_error reports
GE_ERR_DEVICE_CHECK. The ragged, odd-shape and pair-tile GEMM tests, the
split-K and stream-K tests and the decode-stack tests run against it in a child process
(the binding picks the library when it is first loaded)."""
import os
import subprocess
import sys

import pytest

import gemm_epilogues_gb300 as ge

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def debug_lib():
    from gemm_epilogues_gb300 import build
    return build.build(debug=True)


def test_normal_build_has_no_checks_and_probe_is_silent():
    assert not ge.ge_debug_checks()
    with ge.Plan(64, 64, 64, ge.GE_EPI_BIAS) as p:
        assert ge.ge_debug_check_probe(p.handle) == ge.GE_OK
        assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK


def _child(code: str):
    env = dict(os.environ, GE_DEBUG_LIB="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    return r.stdout


def test_checking_build_reports_a_failed_check(debug_lib):
    out = _child(
        "import gemm_epilogues_gb300 as ge\n"
        "assert ge.ge_debug_checks()\n"
        "with ge.Plan(64, 64, 64, ge.GE_EPI_BIAS) as p:\n"
        "    assert ge.ge_debug_check_probe(p.handle) == ge.GE_OK\n"
        "    s = ge.ge_get_last_device_error(p.handle)\n"
        "    assert s == ge.GE_ERR_DEVICE_CHECK, s\n"
        "    assert ge.ge_get_last_device_error(p.handle) == ge.GE_OK\n"
        "print('probe ok')\n")
    assert "probe ok" in out


def test_ragged_pair_split_and_chain_tests_pass_under_checks(debug_lib):
    """Every case checks ge_get_last_device_error, so a failed device check
    fails the case."""
    sel = ("ragged or pair_tiles or 128_wide or stage_panels or split or whole or exact_integer "
           "or every_epilogue or gemv or chain or stream_k or producer")
    out = _child(
        "import sys, pytest\n"
        "import gemm_epilogues_gb300 as ge\n"
        "assert ge.ge_debug_checks()\n"
        f"sys.exit(pytest.main(['-q', '-m', 'gpu', '-p', 'no:cacheprovider', '-k', {sel!r}, "
        "'tests/test_gemm_gpu.py', 'tests/test_chain_gpu.py', 'tests/test_stream_k_gpu.py']))\n")
    assert " passed" in out and " failed" not in out, out[-2000:]
