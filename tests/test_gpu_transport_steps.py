"""The ring transport's GPU side on one GPU: context_long_sequence_gb300.transport
runs its forward and backward schedules with a loopback communicator (one
process holding the whole ring, each "send" a copy into the spare buffer)
and the library's per-step entry points (cp_attn_fwd_step, cp_merge_lse,
cp_attn_bwd_delta, cp_attn_bwd_step), each chunk in its own buffer as a
receiving GPU would hold it.  Results are compared element by element with
the oracle, and with the fused single-launch entry points."""
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
    ("ring_R4_zigzag_docs_d128", 1024, 4, 2, 128, 1, 4, 1, [0, 300, 301, 1024], 1.0),
    ("usp_U2xR3_contig_d64", 1536, 8, 4, 64, 2, 3, 0, None, 1.0),
    ("ring_R8_zigzag_kscale_d128", 2048, 8, 2, 128, 1, 8, 1, None, 0.5),
    ("usp_U2xR2_zigzag_docs_d128", 1024, 8, 2, 128, 2, 2, 1, [0, 500, 1024], 1.0),
]


def _head_sharded(cpa, plan, x, H, elem_bytes=2):
    """[R][U][T][H/U][d] head-sharded copy of a sequence-sharded tensor
    (the Ulysses exchange; with U == 1 just a reshaped view)."""
    R, U, T, d = plan.R, plan.U, plan.L // plan.R, plan.d
    if U == 1:
        return x.view(R, 1, T, H, d)
    out = torch.empty(R, U, T, H // U, d, dtype=x.dtype, device=x.device)
    cpa.ulysses_reshard_batch(plan, [(cpa.CP_SEQ_TO_HEAD, cpa.CP_TOKEN_MAJOR, H, d, elem_bytes, x, out)])
    return out


def _to_seq(cpa, plan, xh, H, elem_bytes):
    """Inverse of _head_sharded."""
    R, U, T, d = plan.R, plan.U, plan.L // plan.R, plan.d
    if U == 1:
        return xh.reshape(R * T, H, d)
    out = torch.empty(R * T, H, d, dtype=xh.dtype, device=xh.device)
    cpa.ulysses_reshard_batch(plan, [(cpa.CP_HEAD_TO_SEQ, cpa.CP_TOKEN_MAJOR, H, d, elem_bytes, xh, out)])
    return out


def _lse_to_seq(cpa, plan, lh):
    R, U, T = plan.R, plan.U, plan.L // plan.R
    if U == 1:
        return lh.reshape(R, plan.Hq, T)
    out = torch.empty(plan.P, plan.Hq, plan.n, dtype=torch.float32, device=lh.device)
    cpa.ulysses_reshard_batch(plan, [(cpa.CP_HEAD_TO_SEQ, cpa.CP_HEAD_MAJOR, plan.Hq, 1, 4, lh, out)])
    return out


def _lse_head(cpa, plan, lse):
    R, U, T = plan.R, plan.U, plan.L // plan.R
    if U == 1:
        return lse.view(R, 1, plan.Hq, T)
    out = torch.empty(R, U, plan.Hq // U, T, dtype=torch.float32, device=lse.device)
    cpa.ulysses_reshard_batch(plan, [(cpa.CP_SEQ_TO_HEAD, cpa.CP_HEAD_MAJOR, plan.Hq, 1, 4, lse, out)])
    return out


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_transport_forward_and_backward_on_one_gpu(cpa, case):
    import gpu_harness as gh
    from context_long_sequence_gb300 import transport as tr
    name, L, Hq, Hkv, d, U, R, layout, docs, ks = case
    inp = workloads.make_inputs(L, Hq, Hkv, d, zlib.crc32(name.encode()) % 1000, k_scale=ks, with_do=True)
    plan = cpa.Plan(L, Hq, Hkv, d, ulysses_degree=U, ring_degree=R, layout=layout, doc_offsets=docs)
    idx = torch.from_numpy(plan.index_map().astype(np.int64))
    q, k, v, do = (inp[n][idx].contiguous().cuda() for n in ("q", "k", "v", "do"))
    T = L // R
    qh = _head_sharded(cpa, plan, q, Hq)
    kh = _head_sharded(cpa, plan, k, Hkv)
    vh = _head_sharded(cpa, plan, v, Hkv)
    kern = tr.CudaRingKernels(plan)
    place = tr.RingPlacement(R=R, U=U, world=1, rank=0)
    comm = tr.LocalComm()

    # Forward: every chunk in its own buffer, rotated through the ring.
    Q = [qh[r] for r in range(R)]
    KV = [(kh[r].clone(), vh[r].clone()) for r in range(R)]
    o_out = [torch.empty_like(Q[r]) for r in range(R)]
    lse_out = [torch.empty(U, Hq // U, T, dtype=torch.float32, device="cuda") for _ in range(R)]
    tr.ring_forward(comm, kern, place, Q, KV, o_out, lse_out)
    assert cpa.cp_get_status() == 0
    o_seq = _to_seq(cpa, plan, torch.stack(o_out), Hq, 2)
    lse_seq = _lse_to_seq(cpa, plan, torch.stack(lse_out).contiguous())
    O, LSE = gh.from_slots(plan, o_seq, lse_seq, idx)
    O_ref, LSE_ref = oracle.attention(inp["q"], inp["k"], inp["v"], offsets=docs)
    gh.assert_close(O.numpy(), LSE.numpy(), O_ref, LSE_ref, name + " transport fwd", bf16_out=True)
    # Beside the single-launch forward (fused merge): the two round P to bf16
    # against different running maxima, so they agree within the workload
    # bounds, not bit for bit; LSE is not rounded to bf16.
    o_f = torch.empty_like(q)
    lse_f = torch.empty(plan.P, Hq, plan.n, dtype=torch.float32, device="cuda")
    cpa.cp_attn_fwd(plan, q, k, v, o_f, lse_f, cpa.alloc_workspace(plan))
    diff = (o_seq.float() - o_f.float()).abs()
    assert float(diff.max()) <= gh.O_MAX_ABS and float(diff.mean()) <= gh.O_MEAN_ABS, float(diff.max())
    assert float((lse_seq - lse_f).abs().max()) <= 1e-5

    # Backward from the single-launch forward's O and LSE.
    oh = _head_sharded(cpa, plan, o_f, Hq)
    doh = _head_sharded(cpa, plan, do, Hq)
    lh = _lse_head(cpa, plan, lse_f)
    dq_out = [torch.empty(U, T, Hq // U, d, dtype=torch.float32, device="cuda") for _ in range(R)]
    KV = [(kh[r].clone(), vh[r].clone()) for r in range(R)]
    dkv = tr.ring_backward(comm, kern, place, Q, KV, [oh[r] for r in range(R)], [lh[r] for r in range(R)],
                           [doh[r] for r in range(R)], dq_out)
    assert cpa.cp_get_status() == 0
    dq_seq = _to_seq(cpa, plan, torch.stack(dq_out), Hq, 4)
    dk_seq = _to_seq(cpa, plan, torch.stack([x[0] for x in dkv]).contiguous(), Hkv, 4)
    dv_seq = _to_seq(cpa, plan, torch.stack([x[1] for x in dkv]).contiguous(), Hkv, 4)
    got = []
    for t in (dq_seq, dk_seq, dv_seq):
        g = torch.empty(t.shape, dtype=torch.float32)
        g[idx] = t.cpu()
        got.append(g.numpy())
    _, _, dq_r, dk_r, dv_r = oracle.attention_bwd(inp["q"].double().numpy(), inp["k"].double().numpy(),
                                                  inp["v"].double().numpy(), inp["do"].double().numpy(),
                                                  offsets=docs)
    gh.assert_grads_close(got, [dq_r, dk_r, dv_r], name + " transport bwd")
    # Beside the single-launch backward: the same products, summed per step.
    dq_f = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    dk_f = torch.empty(k.shape, dtype=torch.float32, device="cuda")
    dv_f = torch.empty(v.shape, dtype=torch.float32, device="cuda")
    cpa.cp_attn_bwd(plan, q, k, v, o_f, lse_f, do, dq_f, dk_f, dv_f, cpa.alloc_workspace(plan, cpa.CP_OP_BWD))
    for a_, b_ in ((dq_seq, dq_f), (dk_seq, dk_f), (dv_seq, dv_f)):
        assert float((a_ - b_).abs().max()) <= 1e-4 * max(1.0, float(b_.abs().max())), float((a_ - b_).abs().max())


def test_step_entries_reject_bad_arguments(cpa):
    plan = cpa.Plan(1024, 4, 2, 128, ring_degree=4, layout=1)
    z = torch.zeros(1024 * 4 * 128, dtype=torch.bfloat16, device="cuda")
    f = torch.zeros(1024 * 4 * 128, dtype=torch.float32, device="cuda")
    for rank, step in ((4, 0), (-1, 0), (0, 4), (0, -1)):
        with pytest.raises(cpa.CPError) as e:
            cpa.cp_attn_fwd_step(plan, rank, step, z, z, z, f, f)
        assert e.value.code == cpa.CP_ERR_INVALID_ARG
        with pytest.raises(cpa.CPError) as e:
            cpa.cp_attn_bwd_step(plan, rank, step, z, z, f, z, z, f, f, f)
        assert e.value.code == cpa.CP_ERR_INVALID_ARG
    ag = cpa.Plan(1024, 4, 2, 128, ring_degree=4, layout=1, kv_exchange=cpa.CP_KV_ALLGATHER)
    with pytest.raises(cpa.CPError) as e:
        cpa.cp_attn_fwd_step(ag, 0, 0, z, z, z, f, f)
    assert e.value.code == cpa.CP_ERR_UNSUPPORTED
