"""GPU parity of the forward path against the CPU oracle, element by element,
at sizes the oracle finishes in seconds (several 128-row tiles, ragged tails,
documents whose boundaries fall inside tiles, GQA, Ulysses, USP and the
emit-partials + merge path), plus reshard and merge bit-exactness and
run-to-run determinism."""
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


def _inputs(L, Hq, Hkv, d, seed):
    return workloads.make_inputs(L, Hq, Hkv, d, seed)


CASES = [
    # name, L, Hq, Hkv, d, U, R, layout, docs, emit_partials
    ("cfg1_ring_L1K_P4_partials", 1024, 4, 4, 64, 1, 4, 0, None, True),
    ("ring_gqa_zigzag_d128", 1536, 8, 2, 128, 1, 3, 1, None, False),
    ("ragged_chunks_d128", 1000, 4, 2, 128, 1, 2, 1, None, False),
    ("docs_inside_tiles", 2048, 4, 1, 128, 1, 2, 1, [0, 300, 301, 1100, 2048], False),
    ("usp_docs", 2048, 8, 4, 128, 2, 2, 1, [0, 777, 2048], False),
    ("ulysses_d64", 1024, 8, 4, 64, 4, 1, 0, None, False),
    ("partials_docs_d64", 768, 4, 2, 64, 1, 2, 1, [0, 100, 500, 768], True),
    ("single_ragged_tile", 72, 2, 1, 128, 1, 1, 0, None, False),
    ("partials_ragged_d128", 600, 4, 4, 128, 1, 3, 0, None, True),
    ("contig_ring_R5_docs", 1280, 4, 2, 64, 1, 5, 0, [0, 5, 6, 640, 1279, 1280], False),
    ("gqa8_zigzag_docs_d128", 1536, 8, 1, 128, 1, 3, 1, [0, 900, 1536], False),
    ("gqa8_usp_U2xR2_d64", 1024, 16, 2, 64, 2, 2, 1, None, False),
]


@pytest.mark.parametrize("out_fp32", [True, False], ids=["o_fp32", "o_bf16"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fwd_matches_oracle(cpa, case, out_fp32):
    import gpu_harness as gh
    name, L, Hq, Hkv, d, U, R, layout, docs, partials = case
    inp = _inputs(L, Hq, Hkv, d, seed=zlib.crc32(name.encode()) % 1000)
    plan = cpa.Plan(L, Hq, Hkv, d, ulysses_degree=U, ring_degree=R, layout=layout, doc_offsets=docs,
                    emit_partials=partials, out_fp32=out_fp32)
    O, LSE = gh.fwd(plan, inp["q"], inp["k"], inp["v"])
    O_ref, LSE_ref = oracle.attention(inp["q"], inp["k"], inp["v"], offsets=docs)
    gh.assert_close(O.numpy(), LSE.numpy(), O_ref, LSE_ref, name, bf16_out=not out_fp32)


JUMP_CASES = [
    # name, L, R, layout, docs, spike keys (position, size) or None for a ramp
    ("spikes_zigzag_R2", 2048, 2, 1, None, [(200, 6.0), (330, 12.0), (777, 18.0), (1500, 24.0)]),
    ("spikes_docs_R1", 1536, 1, 0, [0, 700, 1536], [(100, 8.0), (420, 16.0), (900, 8.0), (1190, 20.0)]),
    ("ramp_R1", 1536, 1, 0, None, None),
]


@pytest.mark.parametrize("case", JUMP_CASES, ids=[c[0] for c in JUMP_CASES])
def test_fwd_running_max_jumps(cpa, case):
    """Scores far above the running max inside wholly visible key tiles, in
    their first or their second 64 keys (spikes), and scores that climb
    steadily along the sequence (ramp).  Every query and key shares a
    component mu, and chosen keys carry a multiple of it, so their score
    exceeds the rest by about 4 log2 units per unit of size."""
    import gpu_harness as gh
    name, L, R, layout, docs, spikes = case
    Hq, Hkv, d = 4, 2, 128
    inp = _inputs(L, Hq, Hkv, d, seed=zlib.crc32(name.encode()) % 1000)
    mu = torch.full((d,), 0.5)
    size = torch.zeros(L)
    if spikes is None:
        size = torch.arange(L, dtype=torch.float32) * (12.0 / L)
    else:
        for pos, a in spikes:
            size[pos] = a
    q = (inp["q"].float() + mu).bfloat16()
    k = (inp["k"].float() + size[:, None, None] * mu).bfloat16()
    plan = cpa.Plan(L, Hq, Hkv, d, ring_degree=R, layout=layout, doc_offsets=docs)
    O, LSE = gh.fwd(plan, q, k, inp["v"])
    O_ref, LSE_ref = oracle.attention(q, k, inp["v"], offsets=docs)
    gh.assert_close(O.numpy(), LSE.numpy(), O_ref, LSE_ref, name, bf16_out=True)


BALANCED_CASES = [
    # name, L, Hq, Hkv, d, U, R, chunks_per_rank, docs, emit_partials
    ("balanced_docs_m3", 1536, 8, 2, 128, 1, 2, 3, [0, 200, 1100, 1536], False),
    ("balanced_usp_m4_d64", 2048, 8, 4, 64, 2, 2, 4, [0, 1500, 2048], False),
    ("balanced_partials_chunk100", 1200, 4, 4, 128, 1, 3, 4, [0, 50, 1200], True),
    ("balanced_one_chunk_R4", 1024, 4, 2, 128, 1, 4, 1, None, False),
    ("balanced_m8_ragged_docs", 2560, 4, 1, 128, 1, 2, 8, [0, 1, 700, 701, 2559, 2560], False),
]


@pytest.mark.parametrize("case", BALANCED_CASES, ids=[c[0] for c in BALANCED_CASES])
def test_fwd_balanced_layout_matches_oracle(cpa, case):
    """Work-balanced chunk layout: chunks of any length (down to below one
    tile), several per rank in position order, with Ulysses, partials and
    documents."""
    import gpu_harness as gh
    name, L, Hq, Hkv, d, U, R, m, docs, partials = case
    inp = _inputs(L, Hq, Hkv, d, seed=zlib.crc32(name.encode()) % 1000)
    plan = cpa.Plan(L, Hq, Hkv, d, ulysses_degree=U, ring_degree=R, layout=cpa.CP_LAYOUT_BALANCED,
                    doc_offsets=docs, emit_partials=partials, out_fp32=True, chunks_per_rank=m)
    O, LSE = gh.fwd(plan, inp["q"], inp["k"], inp["v"])
    O_ref, LSE_ref = oracle.attention(inp["q"], inp["k"], inp["v"], offsets=docs)
    gh.assert_close(O.numpy(), LSE.numpy(), O_ref, LSE_ref, name)


@pytest.mark.parametrize("layout,m,docs", [(1, 2, [0, 300, 1536]), (2, 4, [0, 100, 1000, 1536]), (0, 1, None)])
def test_fwd_rank_by_rank_equals_all_ranks(cpa, layout, m, docs):
    """cp_attn_fwd_rank for every ring rank reproduces cp_attn_fwd_local bit
    for bit, and a rank's call leaves the other ranks' rows untouched."""
    import gpu_harness as gh
    L, Hq, Hkv, d, R = 1536, 4, 2, 128, 3
    inp = _inputs(L, Hq, Hkv, d, seed=50 + layout)
    plan = cpa.Plan(L, Hq, Hkv, d, ring_degree=R, layout=layout, doc_offsets=docs, chunks_per_rank=m)
    idx = torch.from_numpy(plan.index_map().astype(np.int64))
    q, k, v = (gh.to_slots(inp[n], idx).cuda() for n in ("q", "k", "v"))
    o_all = torch.empty_like(q)
    lse_all = torch.empty(R, Hq, L // R, device="cuda")
    cpa.cp_attn_fwd_local(plan, q, k, v, o_all, lse_all)
    o = torch.full_like(q, 7.0)
    lse = torch.full_like(lse_all, 7.0)
    n = L // R
    for r in range(R):
        cpa.cp_attn_fwd_rank(plan, r, q, k, v, o, lse)
        torch.cuda.synchronize()
        assert torch.equal(o[:(r + 1) * n], o_all[:(r + 1) * n]) and torch.equal(lse[:r + 1], lse_all[:r + 1])
        assert (o[(r + 1) * n:] == 7.0).all() and (lse[r + 1:] == 7.0).all()
    assert cpa.cp_get_status() == 0


ALLGATHER_CASES = [
    # name, L, Hq, Hkv, d, R, layout, chunks_per_rank, docs
    ("allgather_contig_R4_docs", 1024, 4, 2, 128, 4, 0, 1, [0, 100, 700, 1024]),
    ("allgather_zigzag_R3_d64", 1536, 8, 2, 64, 3, 1, 2, None),
    ("allgather_balanced_m3_docs", 1536, 4, 1, 128, 2, 2, 3, [0, 5, 900, 1536]),
    ("allgather_ragged", 1000, 4, 4, 128, 2, 1, 2, [0, 499, 1000]),
]


@pytest.mark.parametrize("case", ALLGATHER_CASES, ids=[c[0] for c in ALLGATHER_CASES])
def test_fwd_allgather_matches_oracle(cpa, case):
    """All-gather KV exchange: gather K/V to position order, then every rank's
    queries walk the gathered keys."""
    import gpu_harness as gh
    name, L, Hq, Hkv, d, R, layout, m, docs = case
    inp = _inputs(L, Hq, Hkv, d, seed=zlib.crc32(name.encode()) % 1000)
    plan = cpa.Plan(L, Hq, Hkv, d, ring_degree=R, layout=layout, doc_offsets=docs, chunks_per_rank=m,
                    kv_exchange=cpa.CP_KV_ALLGATHER, out_fp32=True)
    O, LSE = gh.fwd(plan, inp["q"], inp["k"], inp["v"])
    o_ref, lse_ref = oracle.allgather_forward(inp["q"], inp["k"], inp["v"], R, layout, offsets=docs,
                                              chunks_per_rank=m)
    pos = oracle.ring_positions(L, R, layout, docs, m)
    O_ref = np.empty((L, Hq, d))
    O_ref[pos] = o_ref.reshape(L, Hq, d)
    LSE_ref = np.empty((Hq, L))
    LSE_ref[:, pos] = np.concatenate(list(lse_ref), axis=1)
    gh.assert_close(O.numpy(), LSE.numpy(), O_ref, LSE_ref, name)


def test_fwd_allgather_rank_by_rank(cpa):
    """cp_attn_fwd_rank on an all-gather plan (K/V passed gathered, in
    position order) reproduces cp_attn_fwd bit for bit."""
    import gpu_harness as gh
    L, Hq, Hkv, d, R = 1536, 4, 2, 128, 3
    inp = _inputs(L, Hq, Hkv, d, seed=77)
    plan = cpa.Plan(L, Hq, Hkv, d, ring_degree=R, layout=1, doc_offsets=[0, 800, 1536],
                    kv_exchange=cpa.CP_KV_ALLGATHER)
    idx = torch.from_numpy(plan.index_map().astype(np.int64))
    q, k, v = (gh.to_slots(inp[n], idx).cuda() for n in ("q", "k", "v"))
    o_all = torch.empty_like(q)
    lse_all = torch.empty(R, Hq, L // R, device="cuda")
    cpa.cp_attn_fwd(plan, q, k, v, o_all, lse_all, cpa.alloc_workspace(plan))
    kg, vg = inp["k"].cuda(), inp["v"].cuda()
    o = torch.full_like(q, 3.0)
    lse = torch.full_like(lse_all, 3.0)
    for r in range(R):
        cpa.cp_attn_fwd_rank(plan, r, q, kg, vg, o, lse)
    torch.cuda.synchronize()
    assert torch.equal(o, o_all) and torch.equal(lse, lse_all)
    assert cpa.cp_get_status() == 0


@pytest.mark.parametrize("U,R,layout,docs,Hq,Hkv,d", [(4, 1, 0, None, 8, 4, 128), (2, 2, 1, [0, 777, 2048], 8, 4, 128),
                                                      (2, 3, 0, [0, 100, 1536], 4, 2, 64)])
def test_usp_forward_equals_exchanges_around_local(cpa, U, R, layout, docs, Hq, Hkv, d):
    """cp_attn_fwd on a Ulysses/USP plan reads and writes the sequence-sharded
    tensors in place; it must equal, bit for bit, the explicit exchanges
    (ulysses_reshard) around the head-sharded attention (cp_attn_fwd_local),
    whose arithmetic is the same."""
    L = 2048 if R == 2 else 1536 if R == 3 else 1024
    inp = _inputs(L, Hq, Hkv, d, seed=zlib.crc32(f"usp_io_{U}_{R}".encode()) % 1000)
    plan = cpa.Plan(L, Hq, Hkv, d, ulysses_degree=U, ring_degree=R, layout=layout, doc_offsets=docs)
    idx = torch.from_numpy(plan.index_map().astype(np.int64))
    q, k, v = (inp[n][idx].contiguous().cuda() for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(plan.P, Hq, plan.n, dtype=torch.float32, device="cuda")
    cpa.cp_attn_fwd(plan, q, k, v, o, lse, cpa.alloc_workspace(plan))
    T = L // R
    qh = torch.empty(R, U, T, Hq // U, d, dtype=torch.bfloat16, device="cuda")
    kh = torch.empty(R, U, T, Hkv // U, d, dtype=torch.bfloat16, device="cuda")
    vh = torch.empty_like(kh)
    cpa.ulysses_reshard_batch(plan, [(cpa.CP_SEQ_TO_HEAD, cpa.CP_TOKEN_MAJOR, Hq, d, 2, q, qh),
                                     (cpa.CP_SEQ_TO_HEAD, cpa.CP_TOKEN_MAJOR, Hkv, d, 2, k, kh),
                                     (cpa.CP_SEQ_TO_HEAD, cpa.CP_TOKEN_MAJOR, Hkv, d, 2, v, vh)])
    oh = torch.empty_like(qh)
    lh = torch.empty(R, U, Hq // U, T, dtype=torch.float32, device="cuda")
    cpa.cp_attn_fwd_local(plan, qh, kh, vh, oh, lh)
    o2 = torch.empty_like(o)
    lse2 = torch.empty_like(lse)
    cpa.ulysses_reshard_batch(plan, [(cpa.CP_HEAD_TO_SEQ, cpa.CP_TOKEN_MAJOR, Hq, d, 2, oh, o2),
                                     (cpa.CP_HEAD_TO_SEQ, cpa.CP_HEAD_MAJOR, Hq, 1, 4, lh, lse2)])
    torch.cuda.synchronize()
    assert cpa.cp_get_status() == 0
    assert torch.equal(o, o2)
    assert torch.equal(lse, lse2)


def test_fwd_deterministic(cpa):
    import gpu_harness as gh
    inp = _inputs(1536, 8, 2, 128, seed=7)
    plan = cpa.Plan(1536, 8, 2, 128, ring_degree=3, layout=1, doc_offsets=[0, 700, 1536])
    a = gh.fwd(plan, inp["q"], inp["k"], inp["v"])
    b = gh.fwd(plan, inp["q"], inp["k"], inp["v"])
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_partials_equal_fused(cpa):
    """Emit-partials + standalone merge equals the fused ring merge within tolerance."""
    import gpu_harness as gh
    inp = _inputs(1024, 4, 4, 64, seed=11)
    pa = cpa.Plan(1024, 4, 4, 64, ring_degree=4, emit_partials=True)
    pf = cpa.Plan(1024, 4, 4, 64, ring_degree=4, emit_partials=False)
    oa, la = gh.fwd(pa, inp["q"], inp["k"], inp["v"])
    of, lf = gh.fwd(pf, inp["q"], inp["k"], inp["v"])
    assert (oa - of).abs().max().item() <= 1e-2
    assert (la - lf).abs().max().item() <= 1e-4


@pytest.mark.parametrize("R,U,n,H,E,eb", [(2, 4, 48, 8, 128, 2), (1, 4, 64, 32, 64, 2), (3, 2, 10, 4, 3, 4),
                                         (2, 2, 7, 6, 1, 4)])
def test_reshard_bit_exact(cpa, R, U, n, H, E, eb):
    L = R * U * n
    plan = cpa.Plan(L, 8, 8, 64, ulysses_degree=U if 8 % U == 0 else 1, ring_degree=R)
    if plan.U != U:
        pytest.skip("plan shape")
    g = torch.Generator().manual_seed(R * 100 + U)
    dt = torch.int16 if eb == 2 else torch.int32
    x = torch.randint(-30000, 30000, (R, U, n, H, E), generator=g).to(dt)
    xd = x.cuda()
    y = torch.empty(R, U, U * n, H // U, E, dtype=dt, device="cuda")
    cpa.ulysses_reshard(plan, cpa.CP_SEQ_TO_HEAD, cpa.CP_TOKEN_MAJOR, H, E, eb, xd, y)
    ref = np.stack([oracle.ulysses_seq_to_head(x[r].numpy(), U) for r in range(R)])
    assert np.array_equal(y.cpu().numpy(), ref)
    back = torch.empty_like(xd)
    cpa.ulysses_reshard(plan, cpa.CP_HEAD_TO_SEQ, cpa.CP_TOKEN_MAJOR, H, E, eb, y, back)
    assert torch.equal(back, xd)
    # head-major (LSE) direction
    lse = torch.randn(R, U, H, n, generator=g)
    lh = torch.empty(R, U, H // U, U * n, device="cuda")
    cpa.ulysses_reshard(plan, cpa.CP_SEQ_TO_HEAD, cpa.CP_HEAD_MAJOR, H, 1, 4, lse.cuda(), lh)
    lb = torch.empty(R, U, H, n, device="cuda")
    cpa.ulysses_reshard(plan, cpa.CP_HEAD_TO_SEQ, cpa.CP_HEAD_MAJOR, H, 1, 4, lh, lb)
    assert torch.equal(lb.cpu(), lse)
    ref_l = np.stack([oracle.ulysses_lse_head_to_seq(lh[r].cpu().numpy(), U) for r in range(R)])
    assert np.array_equal(ref_l, lse.numpy())


@pytest.mark.parametrize("R,U,n", [(2, 4, 48), (3, 2, 10), (1, 4, 4096)])
def test_reshard_batch_equals_single_calls(cpa, R, U, n):
    """One batched launch (Q, K, V and an odd-sized tensor that needs 4-byte
    words, then O and LSE back) gives the bytes of one call per tensor."""
    L = R * U * n
    plan = cpa.Plan(L, 8, 4, 64, ulysses_degree=U, ring_degree=R)
    g = torch.Generator().manual_seed(7 * R + U)
    q = torch.randint(-30000, 30000, (L, 8, 64), generator=g).to(torch.int16).cuda()
    k = torch.randint(-30000, 30000, (L, 4, 64), generator=g).to(torch.int16).cuda()
    v = torch.randint(-30000, 30000, (L, 4, 64), generator=g).to(torch.int16).cuda()
    odd = torch.randint(-2**30, 2**30, (L, 4, 3), generator=g).to(torch.int32).cuda()   # 12-byte rows
    lse = torch.randn(R * U, 8, n, generator=g).cuda()
    specs = [(8, 64, 2, q), (4, 64, 2, k), (4, 64, 2, v), (4, 3, 4, odd)]
    singles = [torch.empty_like(t) for *_, t in specs]
    batch = [torch.empty_like(t) for *_, t in specs]
    for (H, E, eb, t), y in zip(specs, singles):
        cpa.ulysses_reshard(plan, cpa.CP_SEQ_TO_HEAD, cpa.CP_TOKEN_MAJOR, H, E, eb, t, y)
    cpa.ulysses_reshard_batch(plan, [(cpa.CP_SEQ_TO_HEAD, cpa.CP_TOKEN_MAJOR, H, E, eb, t, y)
                                     for (H, E, eb, t), y in zip(specs, batch)])
    for a, b in zip(singles, batch):
        assert torch.equal(a, b)
    lh1, lh2 = torch.empty_like(lse), torch.empty_like(lse)
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    cpa.ulysses_reshard(plan, cpa.CP_HEAD_TO_SEQ, cpa.CP_TOKEN_MAJOR, 8, 64, 2, singles[0], o1)
    cpa.ulysses_reshard(plan, cpa.CP_HEAD_TO_SEQ, cpa.CP_HEAD_MAJOR, 8, 1, 4, lse, lh1)
    cpa.ulysses_reshard_batch(plan, [(cpa.CP_HEAD_TO_SEQ, cpa.CP_TOKEN_MAJOR, 8, 64, 2, batch[0], o2),
                                     (cpa.CP_HEAD_TO_SEQ, cpa.CP_HEAD_MAJOR, 8, 1, 4, lse, lh2)])
    assert torch.equal(o1, o2) and torch.equal(o2, q)
    assert torch.equal(lh1, lh2)


@pytest.mark.parametrize("n_parts,rows,H,d", [(4, 256, 4, 64), (3, 77, 2, 128), (1, 5, 3, 64), (8, 130, 1, 128)])
def test_merge_matches_oracle(cpa, n_parts, rows, H, d):
    g = torch.Generator().manual_seed(n_parts * 7 + rows)
    o = torch.randn(n_parts, rows, H, d, generator=g)
    lse = torch.randn(n_parts, H, rows, generator=g) * 4
    lse[0, :, ::3] = -float("inf")
    lse[:, 0, 1] = -float("inf")          # a row with every part empty
    o[lse.permute(0, 2, 1)[..., None].expand_as(o) == -float("inf")] = 0.0
    oo = torch.empty(rows, H, d, dtype=torch.bfloat16, device="cuda")
    lo = torch.empty(H, rows, device="cuda")
    cpa.cp_merge_lse(n_parts, rows, H, d, o.cuda(), lse.cuda(), oo, lo)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.merge([(o[p].numpy(), lse[p].numpy()) for p in range(n_parts)])
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(lo.cpu().numpy()), fin)
    assert np.abs(lo.cpu().numpy()[fin] - ref_l[fin]).max() <= 1e-5
    # The merged O is rounded once to bf16 (8 significant bits: unit roundoff
    # 2^-8 with round-to-nearest-even); the fp32 arithmetic before it adds
    # ~1e-6.  Random parts reach |o| ~ 4, where one bf16 half-ulp alone
    # exceeds 1e-2, so the bound is relative.
    err = np.abs(oo.float().cpu().numpy() - ref_o)
    assert (err <= 2.0 ** -8 * np.abs(ref_o) + 1e-5).all(), err.max()


def test_measure_rates(cpa):
    """The rate microbenchmarks behind the secondary bounds return plausible
    figures: tens of exp2 per SM clock, and a bf16 M128 N128 K16 MMA in well
    under a few hundred clocks (64 when the tensor core is fed back to back)."""
    ex2, mma = cpa.cp_measure_rates()
    assert 4.0 <= ex2 <= 128.0, ex2
    assert 32.0 <= mma <= 256.0, mma
    # A completed barrier's check: tens of clocks, far below a wait's limit.
    bc = cpa.cp_measure_barrier_check()
    assert 8.0 <= bc <= 2000.0, bc
    assert cpa.cp_get_status() == 0
