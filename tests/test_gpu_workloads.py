"""GPU parity at the five workloads' full sizes, in the launch configuration
bench.py times (one cp_attn_fwd / cp_attn_bwd call over all emulated ranks),
on sampled outputs the oracle computes one by one: the first and last row of
every chunk and document plus seeded random rows, for query heads that cover
every KV head group and every Ulysses member.  The backward is checked on
sampled dQ rows, on dK/dV of the last keys (whose visible queries are few),
on dK/dV of keys seen by thousands of queries on several ring ranks, and on
the invariants sum_k dV_k = sum_{i, h in group} dO_i (every probability row
sums to one) and sum_k dK_k = 0 (every row of dS sums to zero), which hold
at any size."""
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


# Probabilistic rounding-error bounds for the full-size invariants.  Each
# rounding (to bf16 with unit roundoff u = 2^-8, or an fp32 one) is taken as
# an independent, mean-zero error, the model of Higham and Mary ("A new
# approach to probabilistic rounding error analysis", SIAM J. Sci. Comput.
# 41(5), 2019).  A sum of independent mean-zero terms bounded by b_i stays
# within LAMBDA * sqrt(sum b_i^2) except with probability <= 2 exp(-LAMBDA^2/2)
# (Hoeffding), about 3e-8 for LAMBDA = 6.  Terms that need not be mean zero
# (ex2.approx, the fp32 LSE and the fp32 accumulations) are bounded in the
# worst case by a relative 2^-16, far above their few-ulp size.
U_BF16 = 2.0 ** -8
LAMBDA = 6.0
DET_REL = 2.0 ** -16


def _dv_sum_bound(do_g):
    """sum_k dV_k - sum_{i, h in group} dO_i = sum_i dO_i (sum_k Phat_ik - 1):
    the kernel's P is rounded to bf16 (|error| <= u P), so each query row
    contributes at most u |dO_i| per element.  do_g: [n, Hkv, G, d] fp64."""
    sq = (do_g * do_g).sum(dim=(0, 2))
    ab = do_g.abs().sum(dim=(0, 2))
    return LAMBDA * U_BF16 * sq.sqrt() + DET_REL * ab


def _dk_sum_bound(q_g, do_g, o_g, vmax, scale):
    """sum_k dK_k = scale sum_{i, h in group} q_i X_i with
    X_i = sum_k dShat_ik = dO_i . (O*_i - Ohat_i) + sum_k (rounding of P and dS)
    (in exact arithmetic X_i = dO_i . O_i - D_i = 0).  With ||O* - Ohat|| <=
    u (||Ohat|| + Vmax) (the bf16 output and the bf16 P of the forward) and
    sum_k P_ik |dP_ik - D_i| <= ||dO_i|| (Vmax + ||Ohat_i||),
    |X_i| <= b_i = 3 u ||dO_i|| (Vmax + ||Ohat_i||).
    q_g, do_g, o_g: [n, Hkv, G, d] fp64; vmax [Hkv]: max_k ||v_k||."""
    b = 3 * U_BF16 * do_g.norm(dim=3) * (vmax[None, :, None] + o_g.norm(dim=3))      # [n, Hkv, G]
    rand = (q_g * q_g * (b * b)[..., None]).sum(dim=(0, 2)).sqrt()                 # [Hkv, d]
    det = (q_g.abs() * (b / (3 * U_BF16))[..., None]).sum(dim=(0, 2))
    return scale * (LAMBDA * rand + DET_REL * det)


def _deep_key_rows(w):
    """Keys seen by thousands of queries that sit on several ring ranks: the
    first and last rows of the last three position chunks' tiles (zigzag: the
    chunks of ring ranks 2, 1 and 0; the chunk of rank 1 is visited by rank 0
    at ring step R-1, across the ring's wrap)."""
    c = w.L // (2 * w.ring) if w.layout == workloads.LAYOUT_ZIGZAG else w.L // max(w.ring, 4)
    c = min(c, 4096)
    starts = [w.L - 2 * c, w.L - c]
    rows = {w.L - 2 * c - 1}
    for s0 in starts:
        rows.update({s0, s0 + 1, s0 + 63, s0 + 127, s0 + 128, s0 + c // 2})
    return np.asarray(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("wi", [1, 2], ids=[workloads.WORKLOADS[i].name for i in (1, 2)])
def test_workload_backward_sampled(cpa, wi):
    """The ring backward at the ring workload's size, and the Ulysses
    workload's shapes run backward through the exchanges (its dO drawn after
    V like the ring workload's).  Checked on sampled dQ rows; on dK/dV of the
    last keys (few visible queries) for two KV heads and of keys seen by
    thousands of queries on several ring ranks for one KV head; and on the
    invariants sum_k dV_k = sum_i dO_i and sum_k dK_k = 0 per KV head, whose
    bounds follow from the rounding model above."""
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

    # Invariants at full size, per KV head j and element c.
    G = w.Hq // w.Hkv
    scale = 1.0 / np.sqrt(w.d)
    do_g = do.double().reshape(-1, w.Hkv, G, w.d)
    dv_sum = dv.double().sum(dim=0)                                    # [Hkv, d]
    do_sum = do_g.sum(dim=(0, 2))
    dv_dev = (dv_sum - do_sum).abs()
    dv_tol = _dv_sum_bound(do_g)
    assert (dv_dev <= dv_tol).all(), f"sum dV - sum dO: worst {float((dv_dev / dv_tol).max()):.3f} of the bound"
    vmax = v.double().norm(dim=2).max(dim=0).values                     # [Hkv]
    dk_sum = dk.double().sum(dim=0).abs()
    dk_tol = _dk_sum_bound(q.double().reshape(-1, w.Hkv, G, w.d), do_g, o.double().reshape(-1, w.Hkv, G, w.d),
                           vmax, scale)
    assert (dk_sum <= dk_tol).all(), f"sum dK: worst {float((dk_sum / dk_tol).max()):.3f} of the bound"
    log = os.environ.get("CP_GRAD_ERR_LOG")
    if log:
        import json
        with open(log, "a") as f:
            f.write(json.dumps({"case": w.name, "invariant": "sum dV = sum dO",
                                "worst_over_bound": float((dv_dev / dv_tol).max()),
                                "max_dev": float(dv_dev.max()), "bound_min": float(dv_tol.min())}) + "\n")
            f.write(json.dumps({"case": w.name, "invariant": "sum dK = 0",
                                "worst_over_bound": float((dk_sum / dk_tol).max()),
                                "max_dev": float(dk_sum.max()), "bound_min": float(dk_tol.min())}) + "\n")
    del do_g

    heads = _heads(w.Hq, w.ulysses)
    kv_heads = sorted({h // G for h in heads})
    q_rows = workloads.sample_rows(w.L, _boundaries(w, offsets), 64, seed=w.seed + 1)
    key_rows = np.arange(w.L - 160, w.L, 3)
    deep_rows = _deep_key_rows(w)
    deep_head = kv_heads[-1]
    qr_t = torch.from_numpy(q_rows).to(q.device)
    kr_t = torch.from_numpy(key_rows).to(q.device)
    dr_t = torch.from_numpy(deep_rows).to(q.device)
    got_dq = dq[slot_of[qr_t]][:, heads].cpu().numpy()
    got_dk = dk[slot_of[kr_t]][:, kv_heads].cpu().numpy()
    got_dv = dv[slot_of[kr_t]][:, kv_heads].cpu().numpy()
    deep_dk = dk[slot_of[dr_t]][:, [deep_head]].cpu().numpy()
    deep_dv = dv[slot_of[dr_t]][:, [deep_head]].cpu().numpy()
    cpu = {n: g[n].cpu() for n in ("q", "k", "v", "do")}
    del q, k, v, o, lse, do, dq, dk, dv, g
    torch.cuda.empty_cache()
    ref_dq, ref_dk, ref_dv = oracle.attention_bwd_rows(cpu["q"], cpu["k"], cpu["v"], cpu["do"], q_rows=q_rows,
                                                       key_rows=key_rows, offsets=offsets, q_heads=heads,
                                                       kv_heads=kv_heads)
    gh.assert_grads_close([got_dq, got_dk, got_dv], [ref_dq, ref_dk, ref_dv], w.name)
    _, ref_ddk, ref_ddv = oracle.attention_bwd_rows(cpu["q"], cpu["k"], cpu["v"], cpu["do"], key_rows=deep_rows,
                                                    offsets=offsets, kv_heads=[deep_head])
    gh.assert_grads_close([np.zeros((0, 1, w.d)), deep_dk, deep_dv], [np.zeros((0, 1, w.d)), ref_ddk, ref_ddv],
                          w.name + " (keys seen by thousands of queries)")
