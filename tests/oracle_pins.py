"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` takes the oracle module and raises AssertionError on a
mismatch, so the same pins can be run against deliberately broken copies of
the oracle (see test_oracle_mutations.py) to show that they catch plausible
mistakes.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_examples.json")


def _rand(shape, seed):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape)


def _sdpa_reference(q, k, v, mask, scale):
    """torch's fp64 CPU scaled_dot_product_attention with an explicit mask."""
    L, Hq, d = q.shape
    G = Hq // k.shape[1]
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]                       # [1,Hq,L,d]
    kt = torch.from_numpy(k).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    m = torch.from_numpy(mask)[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


def _lse_reference(q, k, mask, scale):
    """scipy's logsumexp over the visible scores, per head."""
    from scipy.special import logsumexp
    L, Hq, d = q.shape
    G = Hq // k.shape[1]
    out = np.empty((Hq, L))
    for h in range(Hq):
        s = scale * np.einsum("id,kd->ik", q[:, h], k[:, h // G])
        out[h] = logsumexp(np.where(mask, s, -np.inf), axis=1)
    return out


def _explicit_mask(L, offsets):
    ii, kk = np.meshgrid(np.arange(L), np.arange(L), indexing="ij")
    m = kk <= ii
    if offsets is not None:
        doc = np.zeros(L, dtype=np.int64)
        for a, b in zip(offsets[:-1], offsets[1:]):
            doc[a:b] = a
        m &= doc[ii] == doc[kk]
    return m


# ---------------------------------------------------------------- attention


def pin_library_sdpa(orc):
    """GQA causal and document-masked attention vs torch's SDPA (fp64)."""
    for (L, Hq, Hkv, d, offs, seed) in [(37, 4, 2, 8, None, 1), (50, 6, 3, 16, [0, 7, 8, 31, 50], 2),
                                        (64, 4, 4, 4, [0, 64], 3)]:
        q, k, v = _rand((L, Hq, d), seed), _rand((L, Hkv, d), seed + 10), _rand((L, Hkv, d), seed + 20)
        scale = 1.0 / math.sqrt(d)
        mask = _explicit_mask(L, offs)
        O, LSE = orc.attention(q, k, v, offsets=offs)
        np.testing.assert_allclose(O, _sdpa_reference(q, k, v, mask, scale), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(LSE, _lse_reference(q, k, mask, scale), rtol=1e-12, atol=1e-12)


def pin_golden(orc):
    """Hand-derived closed-form examples (tests/golden/closed_form_examples.json)."""
    g = json.load(open(GOLDEN))
    for key in ("causal", "documents"):
        e = g[key]
        q = np.array(e["q"]).reshape(-1, 1, 1)
        k = np.array(e["k"]).reshape(-1, 1, 1)
        v = np.array(e["v"]).reshape(-1, 1, 1)
        O, LSE = orc.attention(q, k, v, offsets=e["doc_offsets"], scale=e["scale"])
        np.testing.assert_allclose(O[:, 0, 0], e["O"], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(LSE[0], e["LSE"], rtol=1e-13, atol=1e-13)
    e = g["merge"]
    a = (np.full((1, 1, 1), e["a"]["O"]), np.full((1, 1), e["a"]["LSE"]))
    b = (np.full((1, 1, 1), e["b"]["O"]), np.full((1, 1), e["b"]["LSE"]))
    o, lse = orc.merge([a, b])
    np.testing.assert_allclose([o.item(), lse.item()], [e["O"], e["LSE"]], rtol=1e-13)
    empty = (np.zeros((1, 1, 1)), np.full((1, 1), -np.inf))
    o2, lse2 = orc.merge([empty, a, empty])
    np.testing.assert_allclose([o2.item(), lse2.item()], [e["a"]["O"], e["a"]["LSE"]], rtol=1e-13)


def pin_first_row_of_document(orc):
    """Row 0 of every document sees only itself: O = v_start, LSE = s_start,start."""
    L, Hq, Hkv, d = 40, 4, 2, 8
    offs = [0, 5, 6, 23, 40]
    q, k, v = _rand((L, Hq, d), 5), _rand((L, Hkv, d), 6), _rand((L, Hkv, d), 7)
    O, LSE = orc.attention(q, k, v, offsets=offs)
    G = Hq // Hkv
    for s in offs[:-1]:
        for h in range(Hq):
            np.testing.assert_allclose(O[s, h], v[s, h // G], rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(LSE[h, s], np.dot(q[s, h], k[s, h // G]) / math.sqrt(d), rtol=1e-12)


def pin_zero_query(orc):
    """Q = 0: uniform weights, O_i = mean of visible v, LSE_i = ln(#visible)."""
    L, Hq, Hkv, d = 33, 2, 1, 4
    offs = [0, 10, 33]
    q = np.zeros((L, Hq, d))
    k, v = _rand((L, Hkv, d), 8), _rand((L, Hkv, d), 9)
    O, LSE = orc.attention(q, k, v, offsets=offs)
    for i in range(L):
        s = 0 if i < 10 else 10
        np.testing.assert_allclose(O[i, 0], v[s:i + 1, 0].mean(axis=0), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(LSE[:, i], math.log(i - s + 1), rtol=1e-13, atol=1e-14)


def pin_constant_v(orc):
    """Constant V gives O = V at every row (weights sum to one)."""
    L, Hq, Hkv, d = 29, 4, 2, 8
    q, k = _rand((L, Hq, d), 10), 3.0 * _rand((L, Hkv, d), 11)
    c = _rand((1, Hkv, d), 12)
    v = np.repeat(c, L, axis=0)
    O, _ = orc.attention(q, k, v, offsets=[0, 3, 29])
    G = Hq // Hkv
    for h in range(Hq):
        np.testing.assert_allclose(O[:, h], np.repeat(c[:, h // G], L, axis=0), rtol=1e-12, atol=1e-12)


def pin_brute_force_loops(orc):
    """Tiny case against scalar Python loops over the definition."""
    L, Hq, Hkv, d = 9, 2, 1, 3
    q, k, v = _rand((L, Hq, d), 13), _rand((L, Hkv, d), 14), _rand((L, Hkv, d), 15)
    O, LSE = orc.attention(q, k, v, offsets=[0, 4, 9])
    for h in range(Hq):
        for i in range(L):
            s0 = 0 if i < 4 else 4
            w = [math.exp(sum(q[i, h, c] * k[j, 0, c] for c in range(d)) / math.sqrt(d)) for j in range(s0, i + 1)]
            z = sum(w)
            for c in range(d):
                ref = sum(w[j - s0] * v[j, 0, c] for j in range(s0, i + 1)) / z
                assert abs(O[i, h, c] - ref) < 1e-12
            assert abs(LSE[h, i] - math.log(z)) < 1e-12


def pin_document_mask_is_separate_attention(orc):
    """Document-masked attention equals attention run on each document alone."""
    L, Hq, Hkv, d = 48, 4, 2, 8
    offs = [0, 11, 12, 30, 48]
    q, k, v = _rand((L, Hq, d), 16), _rand((L, Hkv, d), 17), _rand((L, Hkv, d), 18)
    O, LSE = orc.attention(q, k, v, offsets=offs)
    for a, b in zip(offs[:-1], offs[1:]):
        o, l = orc.attention(q[a:b], k[a:b], v[a:b])
        np.testing.assert_allclose(O[a:b], o, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(LSE[:, a:b], l, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- CP restatement


def pin_ring_equals_full(orc):
    """Ring CP (any R, contiguous or zigzag, with or without documents)
    equals full attention; a one-chunk ring is full attention."""
    L, Hq, Hkv, d = 48, 4, 2, 8
    q, k, v = _rand((L, Hq, d), 19), _rand((L, Hkv, d), 20), _rand((L, Hkv, d), 21)
    for offs in (None, [0, 5, 29, 48]):
        O, LSE = orc.attention(q, k, v, offsets=offs)
        for R, layout in [(1, 0), (4, 0), (3, 1), (4, 1), (2, 1)]:
            o, lse = orc.ring_forward(q, k, v, R, layout, offsets=offs)
            pos = orc.ring_positions(L, R, layout)
            n = L // R
            np.testing.assert_allclose(o.reshape(L, Hq, d), O[pos], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(np.concatenate(list(lse), axis=1), LSE[:, pos], rtol=1e-12, atol=1e-12)
            assert o.shape == (R, n, Hq, d)


def pin_usp_equals_full(orc):
    """USP (Ulysses groups x ring) equals full attention."""
    L, Hq, Hkv, d = 64, 8, 4, 4
    q, k, v = _rand((L, Hq, d), 22), _rand((L, Hkv, d), 23), _rand((L, Hkv, d), 24)
    for offs in (None, [0, 13, 64]):
        O, LSE = orc.attention(q, k, v, offsets=offs)
        for U, R, layout in [(2, 2, 1), (4, 1, 0), (2, 4, 1), (4, 2, 0)]:
            o, lse = orc.usp_forward(q, k, v, U, R, layout, offsets=offs)
            pos = orc.ring_positions(L, R, layout)
            np.testing.assert_allclose(o.reshape(L, Hq, d), O[pos], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(np.concatenate(list(lse), axis=1), LSE[:, pos], rtol=1e-12, atol=1e-12)


def pin_merge_order_independent(orc):
    """Merging disjoint-key partials gives the same result in any order and
    grouping; the empty partial is the identity."""
    n, H, d = 5, 2, 3
    rng = np.random.default_rng(25)
    parts = []
    for i in range(4):
        lse = rng.standard_normal((H, n)) * 3
        if i == 2:
            lse[0, 1] = -np.inf
        o = rng.standard_normal((n, H, d))
        o[1, 0] = 0.0 if i == 2 else o[1, 0]
        parts.append((o, lse))
    ref_o, ref_l = orc.merge(parts)
    for perm in ([3, 1, 0, 2], [2, 3, 1, 0], [1, 0, 3, 2]):
        o, l = orc.merge([parts[p] for p in perm])
        np.testing.assert_allclose(o, ref_o, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(l, ref_l, rtol=1e-12, atol=1e-13)
    left = orc.merge([orc.merge(parts[:2]), orc.merge(parts[2:])])
    np.testing.assert_allclose(left[0], ref_o, rtol=1e-12, atol=1e-13)
    empty = (np.zeros((n, H, d)), np.full((H, n), -np.inf))
    o, l = orc.merge([empty, parts[0], empty])
    np.testing.assert_allclose(o, parts[0][0], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(l, parts[0][1], rtol=1e-13)
    o, l = orc.merge([empty, empty])
    assert np.all(o == 0) and np.all(np.isneginf(l))
    # Direct: the merge of weighted means is the weighted mean of the union.
    w = rng.random((2, 6)) + 0.1
    x = rng.standard_normal((2, 6))
    pa = (np.full((1, 1, 1), (w[0] * x[0]).sum() / w[0].sum()), np.full((1, 1), math.log(w[0].sum())))
    pb = (np.full((1, 1, 1), (w[1] * x[1]).sum() / w[1].sum()), np.full((1, 1), math.log(w[1].sum())))
    o, l = orc.merge([pa, pb])
    np.testing.assert_allclose(o.item(), (w * x).sum() / w.sum(), rtol=1e-13)
    np.testing.assert_allclose(l.item(), math.log(w.sum()), rtol=1e-13)


def pin_reshard(orc):
    """Ulysses reshard: inverse-reshard restores the input bit-exactly; each
    member holds the full group sequence, in group order, of its own
    contiguous block of heads; LSE follows the same map."""
    U, n, H, d = 4, 3, 8, 2
    x = np.arange(U * n * H * d, dtype=np.int64).reshape(U, n, H, d)
    y = orc.ulysses_seq_to_head(x, U)
    assert y.shape == (U, U * n, H // U, d)
    assert np.array_equal(orc.ulysses_head_to_seq(y, U), x)
    # Decode each element's (rank, token, head) from its unique code.
    for u in range(U):
        heads = set()
        for i in range(U * n):
            for hl in range(H // U):
                code = y[u, i, hl, 0]
                s, rem = divmod(code, n * H * d)
                t, rem = divmod(rem, H * d)
                h = rem // d
                assert s * n + t == i          # group order of tokens
                heads.add(h)
        assert heads == set(range(u * H // U, (u + 1) * H // U))
    lse = np.arange(U * H * n, dtype=np.int64).reshape(U, H, n)
    # forward map of LSE written out independently: member u, head hl, token s*n+t
    lse_h = np.empty((U, H // U, U * n), dtype=np.int64)
    for u in range(U):
        for s in range(U):
            lse_h[u, :, s * n:(s + 1) * n] = lse[s, u * H // U:(u + 1) * H // U, :]
    assert np.array_equal(orc.ulysses_lse_head_to_seq(lse_h, U), lse)


def pin_index_maps(orc):
    """Index maps are permutations; zigzag balances causal work exactly:
    rank r holds chunks r and 2R-1-r, so its visible pairs are
    (r c^2 + c(c+1)/2) + ((2R-1-r) c^2 + c(c+1)/2) = (2R-1) c^2 + c(c+1)."""
    for L, R in [(64, 4), (48, 3), (4096, 8), (24, 1)]:
        for layout in (0, 1):
            p = orc.ring_positions(L, R, layout)
            assert sorted(p.tolist()) == list(range(L))
        c = L // (2 * R)
        work = orc.rank_visible_pairs(L, R, 1)
        assert work == [(2 * R - 1) * c * c + c * (c + 1)] * R
        p = orc.ring_positions(L, R, 1)
        assert p[0] == 0 and p[c] == (2 * R - 1) * c and p[L - 1] == (R + 1) * c - 1
        cont = orc.rank_visible_pairs(L, R, 0)
        n = L // R
        assert cont == [sum(r * n + t + 1 for t in range(n)) for r in range(R)]
    assert orc.visible_pairs(10) == 55
    assert orc.visible_pairs(10, [0, 4, 10]) == 10 + 21


def pin_balanced_layout_golden(orc):
    """The work-balanced layout on hand-worked examples (tests/golden)."""
    path = os.path.join(os.path.dirname(__file__), "golden", "balanced_layout_examples.json")
    for ex in json.load(open(path))["examples"]:
        L, R, m, offs = ex["L"], ex["R"], ex["chunks_per_rank"], ex["offsets"]
        assert orc.chunk_work(L, m * R, offs).tolist() == ex["chunk_work"]
        assert orc.balanced_chunks(L, R, m, offs) == ex["rank_chunks"]
        assert orc.rank_visible_pairs(L, R, 2, offs, m) == ex["rank_work"]
        if "zigzag_rank_work" in ex:
            assert orc.rank_visible_pairs(L, R, 1, offs) == ex["zigzag_rank_work"]


def pin_balanced_layout_structure(orc):
    """Balanced maps are permutations made of whole chunks, m per rank, in
    position order within a rank; the ranks' work adds up to the total
    visible pairs; with two chunks per rank and no documents the greedy rule
    reproduces zigzag exactly (chunk work grows with the chunk index, so the
    last R chunks go to ranks 0..R-1 in order and the first R come back in
    reverse)."""
    for L, R in [(64, 4), (48, 3), (4096, 8), (24, 1)]:
        assert np.array_equal(orc.ring_positions(L, R, 2, None, 2), orc.ring_positions(L, R, 1))
    for L, R, m, offs in [(96, 4, 3, [0, 7, 50, 51, 96]), (120, 5, 2, [0, 60, 120]), (64, 2, 8, None)]:
        p = orc.ring_positions(L, R, 2, offs, m)
        assert sorted(p.tolist()) == list(range(L))
        c = L // (m * R)
        chunks = orc.balanced_chunks(L, R, m, offs)
        assert all(len(x) == m for x in chunks)
        for r in range(R):
            starts = p[r * m * c:(r + 1) * m * c:c]
            assert list(starts) == [j * c for j in chunks[r]]
            assert list(starts) == sorted(starts)
            assert np.array_equal(p[r * m * c:(r + 1) * m * c].reshape(m, c) - starts[:, None],
                                  np.tile(np.arange(c), (m, 1)))
        assert sum(orc.rank_visible_pairs(L, R, 2, offs, m)) == orc.visible_pairs(L, offs)


def pin_ring_balanced_equals_full(orc):
    """Ring and USP CP on the balanced layout equal full attention."""
    L, Hq, Hkv, d = 48, 4, 2, 4
    q, k, v = _rand((L, Hq, d), 40), _rand((L, Hkv, d), 41), _rand((L, Hkv, d), 42)
    for offs in (None, [0, 5, 29, 48]):
        O, LSE = orc.attention(q, k, v, offsets=offs)
        for R, m in [(2, 3), (3, 4), (4, 2)]:
            o, lse = orc.ring_forward(q, k, v, R, 2, offsets=offs, chunks_per_rank=m)
            pos = orc.ring_positions(L, R, 2, offs, m)
            np.testing.assert_allclose(o.reshape(L, Hq, d), O[pos], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(np.concatenate(list(lse), axis=1), LSE[:, pos], rtol=1e-12, atol=1e-12)
        o, lse = orc.usp_forward(q, k, v, 2, 2, 2, offsets=offs, chunks_per_rank=3)
        pos = orc.ring_positions(L, 2, 2, offs, 3)
        np.testing.assert_allclose(o.reshape(L, Hq, d), O[pos], rtol=1e-12, atol=1e-12)


def pin_allgather_equals_full(orc):
    """All-gather CP (every layout, with documents) equals full attention,
    rank by rank in slot order."""
    L, Hq, Hkv, d = 48, 4, 2, 4
    q, k, v = _rand((L, Hq, d), 43), _rand((L, Hkv, d), 44), _rand((L, Hkv, d), 45)
    for offs in (None, [0, 7, 30, 48]):
        O, LSE = orc.attention(q, k, v, offsets=offs)
        for R, layout, m in [(4, 0, 1), (3, 1, 2), (2, 2, 3)]:
            o, lse = orc.allgather_forward(q, k, v, R, layout, offsets=offs, chunks_per_rank=m)
            pos = orc.ring_positions(L, R, layout, offs, m)
            np.testing.assert_allclose(o.reshape(L, Hq, d), O[pos], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(np.concatenate(list(lse), axis=1), LSE[:, pos], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- backward


def pin_backward_finite_differences(orc):
    """Gradients of f = sum(dO * O) against central finite differences."""
    L, Hq, Hkv, d = 7, 4, 2, 3
    offs = [0, 3, 7]
    q, k, v = _rand((L, Hq, d), 26), _rand((L, Hkv, d), 27), _rand((L, Hkv, d), 28)
    do = _rand((L, Hq, d), 29)
    _, _, dq, dk, dv = orc.attention_bwd(q, k, v, do, offsets=offs)
    eps = 1e-6

    def f(q_, k_, v_):
        return float((orc.attention(q_, k_, v_, offsets=offs)[0] * do).sum())

    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd = (f(**{a + "_": b for a, b in args_p.items()}) - f(**{a + "_": b for a, b in args_m.items()})) / (2 * eps)
            assert abs(fd - g[idx]) < 1e-7 * max(1.0, abs(fd)), (name, idx, fd, g[idx])


def pin_backward_autograd(orc):
    """Gradients against torch autograd through fp64 SDPA with an explicit mask."""
    L, Hq, Hkv, d = 21, 4, 2, 8
    offs = [0, 9, 21]
    q, k, v = _rand((L, Hq, d), 30), _rand((L, Hkv, d), 31), 0.5 * _rand((L, Hkv, d), 32)
    do = _rand((L, Hq, d), 33)
    O, LSE, dq, dk, dv = orc.attention_bwd(q, k, v, do, offsets=offs)
    G = Hq // Hkv
    qt = torch.from_numpy(q).requires_grad_()
    kt = torch.from_numpy(k).requires_grad_()
    vt = torch.from_numpy(v).requires_grad_()
    m = torch.from_numpy(_explicit_mask(L, offs))[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(
        qt.permute(1, 0, 2)[None], kt.repeat_interleave(G, 1).permute(1, 0, 2)[None],
        vt.repeat_interleave(G, 1).permute(1, 0, 2)[None], attn_mask=m, scale=1 / math.sqrt(d))
    o = o[0].permute(1, 0, 2)
    (o * torch.from_numpy(do)).sum().backward()
    np.testing.assert_allclose(O, o.detach().numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dv, vt.grad.numpy(), rtol=1e-9, atol=1e-11)


def pin_backward_partials_sum_to_full(orc):
    """The per-ring-step backward contributions, summed over the steps of a
    zigzag ring with documents and GQA (dK/dV accumulated on the chunk),
    equal the plain-definition backward (itself pinned by finite differences
    and autograd)."""
    L, Hq, Hkv, d, R = 36, 4, 2, 8, 3
    offs = [0, 13, 14, 36]
    q, k, v = _rand((L, Hq, d), 51), _rand((L, Hkv, d), 52), _rand((L, Hkv, d), 53)
    do = _rand((L, Hq, d), 54)
    O, LSE, dq_ref, dk_ref, dv_ref = orc.attention_bwd(q, k, v, do, offsets=offs)
    pos = orc.ring_positions(L, R, orc.LAYOUT_ZIGZAG, offs)
    n = L // R
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for r in range(R):
        qi = pos[r * n:(r + 1) * n]
        for s in range(R):
            ki = pos[((r - s) % R) * n:(((r - s) % R) + 1) * n]
            pq, pk, pv = orc.attention_bwd_partial(q[qi], do[qi], O[qi], LSE[:, qi], k[ki], v[ki], qi, ki,
                                                   offsets=offs)
            dq[qi] += pq
            dk[ki] += pk
            dv[ki] += pv
    np.testing.assert_allclose(dq, dq_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, dk_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, dv_ref, rtol=1e-10, atol=1e-12)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


def pin_backward_rows_autograd(orc):
    """Selected gradient rows against torch autograd (fp64 SDPA, explicit mask)."""
    L, Hq, Hkv, d = 23, 4, 2, 8
    offs = [0, 10, 23]
    q, k, v = _rand((L, Hq, d), 34), _rand((L, Hkv, d), 35), _rand((L, Hkv, d), 36)
    do = _rand((L, Hq, d), 37)
    G = Hq // Hkv
    qt = torch.from_numpy(q).requires_grad_()
    kt = torch.from_numpy(k).requires_grad_()
    vt = torch.from_numpy(v).requires_grad_()
    m = torch.from_numpy(_explicit_mask(L, offs))[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(
        qt.permute(1, 0, 2)[None], kt.repeat_interleave(G, 1).permute(1, 0, 2)[None],
        vt.repeat_interleave(G, 1).permute(1, 0, 2)[None], attn_mask=m, scale=1 / math.sqrt(d))
    (o[0].permute(1, 0, 2) * torch.from_numpy(do)).sum().backward()
    qr, kr = [0, 5, 9, 10, 22], [0, 3, 9, 12, 21, 22]
    # Default blocking, and two rows per block (several blocks, a ragged last one).
    for blk in (None, 2):
        dq, dk, dv = orc.attention_bwd_rows(q, k, v, do, q_rows=qr, key_rows=kr, offsets=offs, q_heads=[1, 3],
                                            kv_heads=[1], row_block=blk)
        np.testing.assert_allclose(dq, qt.grad.numpy()[qr][:, [1, 3]], rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(dk, kt.grad.numpy()[kr][:, [1]], rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(dv, vt.grad.numpy()[kr][:, [1]], rtol=1e-9, atol=1e-11)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
