"""GPU parity at the five workloads' full sizes, in the launch configuration
bench.py times (one cp_attn_fwd / cp_attn_bwd call over all emulated ranks),
on sampled outputs the oracle computes one by one: the first and last row of
every chunk and document plus seeded random rows, for query heads that cover
every KV head group and every Ulysses member.  The backward is checked on
sampled dQ rows, on dK/dV of the last keys (whose visible queries are few)
and on the invariant sum_k dV_k = sum_{i, h in group} dO_i, which holds at
any size because every probability row sums to one."""
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


def _heads(Hq, U):
    # One head from each Ulysses member and spread over the KV groups.
    per = Hq // U
    hs = sorted({u * per + (u * 5) % per for u in range(U)} | {0, Hq - 1})
    return hs


def _boundaries(w, offsets):
    c = w.L // (2 * w.ring) if w.layout == workloads.LAYOUT_ZIGZAG else w.L // w.ring
    b = list(range(0, w.L, c))
    if offsets is not None:
        b += [int(x) for x in offsets]
    return b


def _run_fwd(cpa, w, dev="cuda", out_fp32=False, with_do=False):
    offsets = workloads.workload_doc_offsets(w)
    plan = cpa.Plan(w.L, w.Hq, w.Hkv, w.d, ulysses_degree=w.ulysses, ring_degree=w.ring, layout=w.layout,
                    doc_offsets=offsets, emit_partials=w.emit_partials, out_fp32=out_fp32)
    g = workloads.make_inputs(w.L, w.Hq, w.Hkv, w.d, w.seed, device=dev, k_scale=w.k_scale,
                              with_do=w.backward or with_do)
    idx = torch.from_numpy(plan.index_map().astype(np.int64)).to(dev)
    q, k, v = (g[n][idx].contiguous() for n in ("q", "k", "v"))
    o = torch.empty(q.shape, dtype=plan.o_dtype, device=dev)
    lse = torch.empty(plan.P, w.Hq, plan.n, dtype=torch.float32, device=dev)
    ws = cpa.alloc_workspace(plan, device=dev)
    cpa.cp_attn_fwd(plan, q, k, v, o, lse, ws)
    assert cpa.cp_get_status() == 0
    del ws
    slot_of = torch.empty_like(idx)
    slot_of[idx] = torch.arange(w.L, device=dev)
    return plan, offsets, g, (q, k, v, o, lse), slot_of


@pytest.mark.parametrize("out_fp32", [False, True], ids=["o_bf16", "o_fp32"])
@pytest.mark.parametrize("wi", [0, 1, 2, 3, 4], ids=[w.name for w in workloads.WORKLOADS])
def test_workload_forward_sampled(cpa, wi, out_fp32):
    import gpu_harness as gh
    w = workloads.WORKLOADS[wi]
    plan, offsets, g, (q, k, v, o, lse), slot_of = _run_fwd(cpa, w, out_fp32=out_fp32)
    per_head = 256 if w.L <= 65536 else 48
    rows = workloads.sample_rows(w.L, _boundaries(w, offsets), per_head, seed=w.seed)
    if w.L <= 1024:
        rows = np.arange(w.L)
    heads = _heads(w.Hq, w.ulysses)
    rows_t = torch.from_numpy(rows).to(q.device)
    slots = slot_of[rows_t]
    O = o[slots][:, heads].float().cpu().numpy()
    lse_slots = lse.permute(1, 0, 2).reshape(w.Hq, w.L)
    LSE = lse_slots[heads][:, slots].cpu().numpy()
    del q, k, v, o, lse
    cpu = {n: g[n].cpu() for n in ("q", "k", "v")}
    del g
    torch.cuda.empty_cache()
    O_ref, LSE_ref = oracle.attention_rows(cpu["q"], cpu["k"], cpu["v"], rows=rows, offsets=offsets, heads=heads)
    gh.assert_close(O, LSE, O_ref, LSE_ref, w.name, bf16_out=not out_fp32)


@pytest.mark.parametrize("kv_exchange", [0, 1], ids=["ring", "allgather"])
def test_packed_documents_balanced_layout_sampled(cpa, kv_exchange):
    """The packed-document workload (L = 131072, R = 16, seeded documents)
    on the work-balanced layout with 8 chunks per rank, with the ring or the
    all-gather KV exchange: sampled rows against the oracle."""
    import gpu_harness as gh
    w = workloads.WORKLOADS[3]
    offsets = workloads.workload_doc_offsets(w)
    plan = cpa.Plan(w.L, w.Hq, w.Hkv, w.d, ring_degree=w.ring, layout=cpa.CP_LAYOUT_BALANCED, doc_offsets=offsets,
                    chunks_per_rank=8, out_fp32=True, kv_exchange=kv_exchange)
    g = workloads.make_inputs(w.L, w.Hq, w.Hkv, w.d, w.seed, device="cuda", k_scale=w.k_scale)
    idx = torch.from_numpy(plan.index_map().astype(np.int64)).to("cuda")
    q, k, v = (g[n][idx].contiguous() for n in ("q", "k", "v"))
    o = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(plan.P, w.Hq, plan.n, dtype=torch.float32, device="cuda")
    ws = cpa.alloc_workspace(plan)
    cpa.cp_attn_fwd(plan, q, k, v, o, lse, ws)
    assert cpa.cp_get_status() == 0
    del ws
    slot_of = torch.empty_like(idx)
    slot_of[idx] = torch.arange(w.L, device="cuda")
    c = w.L // (8 * w.ring)
    rows = workloads.sample_rows(w.L, list(range(0, w.L, c)) + [int(x) for x in offsets], 48, seed=w.seed + 2)
    heads = _heads(w.Hq, 1)
    rows_t = torch.from_numpy(rows).to("cuda")
    slots = slot_of[rows_t]
    O = o[slots][:, heads].cpu().numpy()
    LSE = lse.permute(1, 0, 2).reshape(w.Hq, w.L)[heads][:, slots].cpu().numpy()
    cpu = {n: g[n].cpu() for n in ("q", "k", "v")}
    del q, k, v, o, lse, g
    torch.cuda.empty_cache()
    O_ref, LSE_ref = oracle.attention_rows(cpu["q"], cpu["k"], cpu["v"], rows=rows, offsets=offsets, heads=heads)
    gh.assert_close(O, LSE, O_ref, LSE_ref, "packed docs, balanced layout")


@pytest.mark.parametrize("wi", [1, 2], ids=[workloads.WORKLOADS[i].name for i in (1, 2)])
def test_workload_backward_sampled(cpa, wi):
    """The ring backward at the ring workload's size, and the Ulysses
    workload's shapes run backward through the exchanges (its dO drawn after
    V like the ring workload's)."""
    import gpu_harness as gh
    w = workloads.WORKLOADS[wi]
    plan, offsets, g, (q, k, v, o, lse), slot_of = _run_fwd(cpa, w, with_do=True)
    idx = torch.from_numpy(plan.index_map().astype(np.int64)).to(q.device)
    do = g["do"][idx].contiguous()
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    dk = torch.empty(k.shape, dtype=torch.float32, device=q.device)
    dv = torch.empty(v.shape, dtype=torch.float32, device=q.device)
    cpa.cp_attn_bwd(plan, q, k, v, o, lse, do, dq, dk, dv, cpa.alloc_workspace(plan, cpa.CP_OP_BWD))
    assert cpa.cp_get_status() == 0

    # Invariant at full size: sum over keys of dV equals the sum of dO over
    # queries and the group's heads.  Bound: each query row contributes
    # sum_k P_ik dO_i with P rounded to bf16 (unit roundoff 2^-8).
    G = w.Hq // w.Hkv
    dv_sum = dv.double().sum(dim=0)                                    # [Hkv, d]
    do_sum = do.double().sum(dim=0).reshape(w.Hkv, G, w.d).sum(dim=1)
    do_abs = do.double().abs().sum(dim=0).reshape(w.Hkv, G, w.d).sum(dim=1)
    assert ((dv_sum - do_sum).abs() <= 2.0 ** -8 * do_abs + 1e-3).all()

    heads = _heads(w.Hq, w.ulysses)
    kv_heads = sorted({h // G for h in heads})
    q_rows = workloads.sample_rows(w.L, _boundaries(w, offsets), 64, seed=w.seed + 1)
    key_rows = np.arange(w.L - 160, w.L, 3)
    qr_t = torch.from_numpy(q_rows).to(q.device)
    kr_t = torch.from_numpy(key_rows).to(q.device)
    got_dq = dq[slot_of[qr_t]][:, heads].cpu().numpy()
    got_dk = dk[slot_of[kr_t]][:, kv_heads].cpu().numpy()
    got_dv = dv[slot_of[kr_t]][:, kv_heads].cpu().numpy()
    cpu = {n: g[n].cpu() for n in ("q", "k", "v", "do")}
    ref_dq, ref_dk, ref_dv = oracle.attention_bwd_rows(cpu["q"], cpu["k"], cpu["v"], cpu["do"], q_rows=q_rows,
                                                       key_rows=key_rows, offsets=offsets, q_heads=heads,
                                                       kv_heads=kv_heads)
    gh.assert_grads_close([got_dq, got_dk, got_dv], [ref_dq, ref_dk, ref_dv], w.name)
