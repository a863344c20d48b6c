"""cp_attn_fwd_noalloc: the allocation-free forward for callers that cannot
call cudaMalloc (a plugin inside a framework that owns the device allocator,
a runtime with a device-memory budget fixed at start-up, a latency-critical
loop that must avoid cudaMalloc's implicit synchronisation).

It runs the same kernels on the same work items as cp_attn_fwd with a
caller workspace, so on two calls in a row (the static scratch keeps the
previous call's contents) its O and LSE must equal cp_attn_fwd's bit for
bit, and both must match the oracle within the workload bounds.  The second
call must not change the device memory in use, neither torch's allocator
count nor the driver's free bytes (the first call may still load a kernel
module lazily).  A problem whose partials exceed the static scratch is
rejected.  This file is collected last so that a failure here does not hide
any other test.
"""
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


# The 1K-token, 4-rank ring workload (d=64) and a ragged d=128 ring with documents.
CASES = [(1024, 4, 4, 64, 4, None, 1000), (600, 4, 2, 128, 3, [0, 250, 600], 3)]


@pytest.mark.parametrize("case", CASES, ids=["L1K_P4_d64", "L600_R3_docs_d128"])
def test_noalloc_matches_workspace_entry_point_and_oracle(cpa, case):
    import gpu_harness as gh
    L, Hq, Hkv, d, R, docs, seed = case
    plan = cpa.Plan(L, Hq, Hkv, d, ring_degree=R, emit_partials=True, doc_offsets=docs)
    inp = workloads.make_inputs(L, Hq, Hkv, d, seed)
    idx = torch.from_numpy(plan.index_map().astype(np.int64))
    q, k, v = (inp[n][idx].contiguous().cuda() for n in ("q", "k", "v"))
    o_ref = torch.empty_like(q)
    lse_ref = torch.empty(plan.P, Hq, plan.n, device="cuda")
    cpa.cp_attn_fwd(plan, q, k, v, o_ref, lse_ref, cpa.alloc_workspace(plan))
    assert cpa.cp_get_status() == 0
    O_orc, LSE_orc = oracle.attention(inp["q"], inp["k"], inp["v"], offsets=docs)
    outs = [(torch.full_like(q, float("nan")), torch.full((plan.P, Hq, plan.n), float("nan"), device="cuda"))
            for _ in range(2)]
    for call, (o, lse) in enumerate(outs):
        torch.cuda.synchronize()
        used0 = torch.cuda.memory_allocated()
        free0, _ = torch.cuda.mem_get_info()
        cpa.cp_attn_fwd_noalloc(plan, q, k, v, o, lse)
        assert cpa.cp_get_status() == 0
        torch.cuda.synchronize()
        if call == 1:
            assert torch.cuda.memory_allocated() == used0, "torch allocation changed during the call"
            assert torch.cuda.mem_get_info()[0] == free0, "device free bytes changed during the call"
        assert torch.equal(o, o_ref), (call, (o.float() - o_ref.float()).abs().max().item())
        assert torch.equal(lse, lse_ref), (call, (lse - lse_ref).abs().max().item())
        O, LSE = gh.from_slots(plan, o, lse, idx)
        gh.assert_close(O.numpy(), LSE.numpy(), O_orc, LSE_orc, f"noalloc call {call}", bf16_out=True)


def test_noalloc_rejects_oversized_and_non_partial_plans(cpa):
    # 4 ranks x 16384 tokens x 4 heads x (64 + 1) floats = 68 MB > 8 MiB.
    big = cpa.Plan(16384, 4, 4, 64, ring_degree=4, emit_partials=True)
    z = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    zf = torch.zeros(1, device="cuda")
    with pytest.raises(cpa.CPError) as e:
        cpa.cp_attn_fwd_noalloc(big, z, z, z, z, zf)
    assert e.value.code == cpa.CP_ERR_WORKSPACE
    fused = cpa.Plan(1024, 4, 4, 64, ring_degree=4, emit_partials=False)
    with pytest.raises(cpa.CPError) as e:
        cpa.cp_attn_fwd_noalloc(fused, z, z, z, z, zf)
    assert e.value.code == cpa.CP_ERR_INVALID_ARG
