"""cp_attn_fwd_noalloc: the allocation-free forward for callers that cannot
call cudaMalloc (a plugin inside a framework that owns the device allocator,
a runtime with a device-memory budget fixed at start-up, a latency-critical
loop that must avoid cudaMalloc's implicit synchronisation).

It must give the same result as cp_attn_fwd with a caller workspace, on two
calls in a row (the static scratch keeps the previous call's contents), and
reject a problem whose partials exceed the static scratch.  This file is
collected last so that a failure here does not hide any other test.
"""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(__file__))

pytestmark = pytest.mark.gpu

import workloads  # noqa: E402


@pytest.fixture(scope="module")
def cpa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import context_long_sequence_gb300 as m
    return m


def _sharded_inputs(plan, seed):
    inp = workloads.make_inputs(plan.L, plan.Hq, plan.Hkv, plan.d, seed)
    idx = torch.from_numpy(plan.index_map().astype(np.int64))
    return [inp[n][idx].contiguous().cuda() for n in ("q", "k", "v")]


def test_noalloc_matches_workspace_entry_point(cpa):
    import gpu_harness as gh
    # The 1K-token, 4-rank ring workload (d=64) and a ragged d=128 ring.
    for (L, Hq, Hkv, d, R, docs, seed) in [(1024, 4, 4, 64, 4, None, 1000), (600, 4, 2, 128, 3, [0, 250, 600], 3)]:
        plan = cpa.Plan(L, Hq, Hkv, d, ring_degree=R, emit_partials=True, doc_offsets=docs)
        q, k, v = _sharded_inputs(plan, seed)
        o_ref = torch.empty_like(q)
        lse_ref = torch.empty(plan.P, Hq, plan.n, device="cuda")
        cpa.cp_attn_fwd(plan, q, k, v, o_ref, lse_ref, cpa.alloc_workspace(plan))
        assert cpa.cp_get_status() == 0
        for call in range(2):
            o = torch.full_like(q, float("nan"))
            lse = torch.full((plan.P, Hq, plan.n), float("nan"), device="cuda")
            cpa.cp_attn_fwd_noalloc(plan, q, k, v, o, lse)
            assert cpa.cp_get_status() == 0
            eo = (o.float() - o_ref.float()).abs()
            el = (lse - lse_ref).abs()
            assert torch.isfinite(o.float()).all()
            assert eo.max().item() <= gh.O_MAX_ABS and eo.mean().item() <= gh.O_MEAN_ABS, (call, eo.max().item())
            assert el.max().item() <= gh.LSE_MAX_ABS, (call, el.max().item())


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
