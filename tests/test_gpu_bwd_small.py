"""GPU parity of the backward (dQ, dK, dV) against the fp64 oracle,
element by element: GQA, zigzag and contiguous rings, ragged chunks, packed
documents whose boundaries fall inside tiles, K scaled by 0.5; and
Ulysses and USP plans (gradients resharded back through the exchanges);
run-to-run determinism (no atomics)."""
import os
import sys
import zlib

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


CASES = [
    # name, L, Hq, Hkv, d, U, R, layout, docs, k_scale
    ("gqa_zigzag_d128", 1024, 4, 2, 128, 1, 2, 1, None, 1.0),
    ("ragged_docs_d64", 1000, 4, 1, 64, 1, 2, 1, [0, 300, 301, 1000], 1.0),
    ("contig_R3_docs_d128", 768, 2, 2, 128, 1, 3, 0, [0, 200, 700, 768], 1.0),
    ("ring_R8_zigzag_kscale", 2048, 8, 2, 128, 1, 8, 1, None, 0.5),
    # Ulysses and USP: gradients pass back through the exchanges.
    ("ulysses_U4_gqa_d128", 1024, 8, 4, 128, 4, 1, 0, None, 1.0),
    ("usp_U2xR2_zigzag_docs_d64", 1536, 8, 2, 64, 2, 2, 1, [0, 500, 520, 1536], 1.0),
    ("usp_U2xR3_ragged_d128", 1440, 4, 2, 128, 2, 3, 0, [0, 711, 1440], 0.5),
    # Eight query heads per KV head (the whole group on one Ulysses member).
    ("gqa8_zigzag_docs_d128", 1536, 8, 1, 128, 1, 3, 1, [0, 900, 1536], 1.0),
    ("gqa8_usp_U2xR2_d64", 1024, 16, 2, 64, 2, 2, 1, None, 1.0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_bwd_matches_oracle(cpa, case):
    import gpu_harness as gh
    name, L, Hq, Hkv, d, U, R, layout, docs, ks = case
    inp = workloads.make_inputs(L, Hq, Hkv, d, zlib.crc32(name.encode()) % 1000, k_scale=ks, with_do=True)
    plan = cpa.Plan(L, Hq, Hkv, d, ulysses_degree=U, ring_degree=R, layout=layout, doc_offsets=docs)
    got = gh.bwd(plan, inp["q"], inp["k"], inp["v"], inp["do"])
    _, _, dq, dk, dv = oracle.attention_bwd(inp["q"].double().numpy(), inp["k"].double().numpy(),
                                            inp["v"].double().numpy(), inp["do"].double().numpy(), offsets=docs)
    gh.assert_grads_close([g.numpy() for g in got], [dq, dk, dv], name)


@pytest.mark.parametrize("U,R,m,docs", [(1, 2, 3, [0, 200, 1100, 1536]), (2, 2, 4, [0, 900, 1536]),
                                        (1, 3, 4, None)])
def test_bwd_balanced_layout(cpa, U, R, m, docs):
    """Backward on the work-balanced chunk layout."""
    import gpu_harness as gh
    L, Hq, Hkv, d = 1536, 8, 2, 128
    inp = workloads.make_inputs(L, Hq, Hkv, d, 40 + U + R + m, with_do=True)
    plan = cpa.Plan(L, Hq, Hkv, d, ulysses_degree=U, ring_degree=R, layout=cpa.CP_LAYOUT_BALANCED,
                    doc_offsets=docs, chunks_per_rank=m)
    got = gh.bwd(plan, inp["q"], inp["k"], inp["v"], inp["do"])
    _, _, dq, dk, dv = oracle.attention_bwd(inp["q"].double().numpy(), inp["k"].double().numpy(),
                                            inp["v"].double().numpy(), inp["do"].double().numpy(), offsets=docs)
    gh.assert_grads_close([g.numpy() for g in got], [dq, dk, dv], f"balanced U{U} R{R} m{m}")


def test_bwd_allgather_plan(cpa):
    """An all-gather plan's backward (dK, dV land in the owners' slots)."""
    import gpu_harness as gh
    L, Hq, Hkv, d = 1024, 4, 2, 128
    docs = [0, 300, 1024]
    inp = workloads.make_inputs(L, Hq, Hkv, d, 61, with_do=True)
    plan = cpa.Plan(L, Hq, Hkv, d, ring_degree=4, layout=1, doc_offsets=docs, kv_exchange=cpa.CP_KV_ALLGATHER)
    got = gh.bwd(plan, inp["q"], inp["k"], inp["v"], inp["do"])
    _, _, dq, dk, dv = oracle.attention_bwd(inp["q"].double().numpy(), inp["k"].double().numpy(),
                                            inp["v"].double().numpy(), inp["do"].double().numpy(), offsets=docs)
    gh.assert_grads_close([g.numpy() for g in got], [dq, dk, dv], "allgather plan")


def test_bwd_deterministic(cpa):
    import gpu_harness as gh
    inp = workloads.make_inputs(1024, 4, 2, 128, 5, with_do=True)
    plan = cpa.Plan(1024, 4, 2, 128, ring_degree=2, layout=1, doc_offsets=[0, 400, 1024])
    a = gh.bwd(plan, inp["q"], inp["k"], inp["v"], inp["do"])
    b = gh.bwd(plan, inp["q"], inp["k"], inp["v"], inp["do"])
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_bwd_with_fp32_o(cpa):
    """The backward reads an fp32 O (plan out_fp32) for D = rowsum(dO * O)."""
    import gpu_harness as gh
    inp = workloads.make_inputs(768, 4, 2, 128, 21, with_do=True)
    plan = cpa.Plan(768, 4, 2, 128, ring_degree=3, layout=1, doc_offsets=[0, 300, 768], out_fp32=True)
    got = gh.bwd(plan, inp["q"], inp["k"], inp["v"], inp["do"])
    _, _, dq, dk, dv = oracle.attention_bwd(inp["q"].double().numpy(), inp["k"].double().numpy(),
                                            inp["v"].double().numpy(), inp["do"].double().numpy(),
                                            offsets=[0, 300, 768])
    gh.assert_grads_close([g.numpy() for g in got], [dq, dk, dv], "fp32 O")


def test_bwd_usp_deterministic_fp32_o(cpa):
    """USP backward with an fp32 O: matches the oracle and repeats bit for bit."""
    import gpu_harness as gh
    docs = [0, 100, 1024]
    inp = workloads.make_inputs(1024, 8, 4, 128, 31, with_do=True)
    plan = cpa.Plan(1024, 8, 4, 128, ulysses_degree=2, ring_degree=2, layout=1, doc_offsets=docs, out_fp32=True)
    a = gh.bwd(plan, inp["q"], inp["k"], inp["v"], inp["do"])
    b = gh.bwd(plan, inp["q"], inp["k"], inp["v"], inp["do"])
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    _, _, dq, dk, dv = oracle.attention_bwd(inp["q"].double().numpy(), inp["k"].double().numpy(),
                                            inp["v"].double().numpy(), inp["do"].double().numpy(), offsets=docs)
    gh.assert_grads_close([g.numpy() for g in a], [dq, dk, dv], "usp fp32 O")
