"""The bounds-checked debug build (libcpattn_debug.so, -DCP_DEBUG).

1. The record routine the checks use writes {CP_ERR_DEVICE_BOUNDS, block,
   line, file id} and skips the access; the context stays usable.
2. The GPU parity suites, run again in a child process against the debug
   library, pass with every check compiled in and leave no record: every
   work item, global index and TMA coordinate of the release path's
   launches stays in bounds on those cases (ragged tails, documents,
   Ulysses, USP, zigzag, balanced, all-gather, emit-partials, backward)."""
import os
import subprocess
import sys

import pytest
import torch

sys.path.insert(0, os.path.dirname(__file__))

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def cpa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import context_long_sequence_gb300 as m
    return m


@pytest.mark.parametrize("block", [0, 37])
def test_bounds_record(cpa, block):
    assert cpa.cp_get_status_detail()[0] == 0
    line = cpa.cp_selftest_bounds(block)
    assert line > 0
    assert cpa.cp_get_status_detail() == (cpa.CP_ERR_DEVICE_BOUNDS, block, line, 1)
    assert cpa.cp_get_status_detail() == (0, 0, 0, 0)  # read and cleared


def test_bounds_record_keeps_first_error(cpa):
    cpa.cp_selftest_wait_timeout(1000)  # records CP_ERR_DEVICE_TIMEOUT first
    cpa.cp_selftest_bounds(3)
    assert cpa.cp_get_status_detail()[0] == cpa.CP_ERR_DEVICE_TIMEOUT


def test_parity_suites_under_debug_build():
    lib = os.path.join(ROOT, "context_long_sequence_gb300", "libcpattn_debug.so")
    if not os.path.exists(lib):
        from context_long_sequence_gb300 import build as b
        b.build()
    env = dict(os.environ, CPATTN_DEBUG="1")
    probe = subprocess.run([sys.executable, "-c", "import context_long_sequence_gb300 as c; print(c.cp_debug_build())"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.stdout.strip() == "True", probe.stdout + probe.stderr
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_gpu_fwd_small.py", "tests/test_gpu_bwd_small.py"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
