"""Device-side failure detection without a GPU fault: a wait on a barrier
that nothing completes runs out after a short limit, records
CP_ERR_DEVICE_TIMEOUT in the status word, and raises the CTA's abort flag so
that its other role leaves too; the kernel returns normally and the next
calls on the same context work."""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(__file__))

pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import workloads  # noqa: E402


@pytest.fixture(scope="module")
def cpa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import context_long_sequence_gb300 as m
    return m


def test_wait_timeout_is_reported_and_context_stays_usable(cpa):
    import gpu_harness as gh
    cpa.cp_get_status()  # clear
    timed_out, left_on_abort, wait_us = cpa.cp_selftest_wait_timeout(20000)  # 20 ms limit
    assert timed_out == 1
    assert left_on_abort == 1
    # The second role left because of the abort flag, long before its own 2 s limit.
    assert 15000 <= wait_us < 1000000, wait_us
    assert cpa.cp_get_status() == cpa.CP_ERR_DEVICE_TIMEOUT
    assert cpa.cp_get_status() == 0  # read and cleared
    # Same context, next call: a small forward still matches the oracle.
    inp = workloads.make_inputs(512, 4, 2, 128, 3)
    plan = cpa.Plan(512, 4, 2, 128, ring_degree=2, layout=1, doc_offsets=[0, 200, 512])
    O, LSE = gh.fwd(plan, inp["q"], inp["k"], inp["v"])
    O_ref, LSE_ref = oracle.attention(inp["q"], inp["k"], inp["v"], offsets=[0, 200, 512])
    gh.assert_close(O.numpy(), LSE.numpy(), O_ref, LSE_ref, "after the self-test", bf16_out=True)


def test_selftest_rejects_bad_limits(cpa):
    for bad in (0, -5, 2000000):
        with pytest.raises(cpa.CPError):
            cpa.cp_selftest_wait_timeout(bad)
