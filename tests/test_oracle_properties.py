"""Property tests of the oracle (CPU, hypothesis): the invariants that make
the context-parallel restatement equal to plain attention hold for randomly
drawn shapes, layouts and document splits, not only for the fixed cases of
the pins.

- Merging normalised partials over disjoint key sets does not depend on the
  order or the grouping, and the empty partial (0, -inf) is its identity.
- The ring forward over any ring degree and token layout, with any packed
  documents, equals full attention.
- Every layout's index map is a permutation of the positions.
- The touched key tiles of the tile-class derivation hold every visible
  (query, key) pair exactly once."""
import math

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from oracle.tiles import tile_classes  # noqa: E402

SETTINGS = settings(max_examples=40, deadline=None, derandomize=True)


@st.composite
def partial_sets(draw):
    n = draw(st.integers(1, 6))
    H = draw(st.integers(1, 3))
    d = draw(st.integers(1, 4))
    k = draw(st.integers(1, 5))
    seed = draw(st.integers(0, 2**31 - 1))
    rng = np.random.default_rng(seed)
    parts = []
    for _ in range(k):
        lse = rng.standard_normal((H, n)) * draw(st.floats(0.1, 20.0))
        empty = rng.random((H, n)) < 0.25
        lse[empty] = -np.inf
        o = rng.standard_normal((n, H, d))
        o[empty.T] = 0.0
        parts.append((o, lse))
    return parts, seed


@SETTINGS
@given(partial_sets())
def test_merge_is_order_and_grouping_free(ps):
    parts, seed = ps
    ref_o, ref_l = oracle.merge(parts)
    perm = np.random.default_rng(seed + 1).permutation(len(parts))
    o, l = oracle.merge([parts[i] for i in perm])
    np.testing.assert_allclose(o, ref_o, rtol=1e-11, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(l), np.isneginf(ref_l))
    fin = np.isfinite(ref_l)
    np.testing.assert_allclose(l[fin], ref_l[fin], rtol=1e-11, atol=1e-12)
    if len(parts) > 1:
        cut = len(parts) // 2
        o2, l2 = oracle.merge([oracle.merge(parts[:cut]), oracle.merge(parts[cut:])])
        np.testing.assert_allclose(o2, ref_o, rtol=1e-11, atol=1e-12)
    n, H, d = parts[0][0].shape
    empty = (np.zeros((n, H, d)), np.full((H, n), -np.inf))
    o3, l3 = oracle.merge([empty] + list(parts) + [empty])
    np.testing.assert_allclose(o3, ref_o, rtol=1e-12, atol=1e-13)


@st.composite
def ring_plans(draw):
    R = draw(st.integers(1, 4))
    layout = draw(st.sampled_from([0, 1, 2]))
    m = {0: 1, 1: 2, 2: draw(st.sampled_from([2, 3, 4]))}[layout]
    chunk = draw(st.integers(1, 6))
    L = R * m * chunk
    n_cuts = draw(st.integers(0, min(3, L - 1)))
    cuts = sorted(draw(st.sets(st.integers(1, L - 1), min_size=n_cuts, max_size=n_cuts))) if L > 1 else []
    docs = [0] + cuts + [L] if cuts else None
    return L, R, layout, m, docs, draw(st.integers(0, 10**6))


@SETTINGS
@given(ring_plans())
def test_ring_forward_equals_full_attention(plan):
    L, R, layout, m, docs, seed = plan
    rng = np.random.default_rng(seed)
    q, k, v = rng.standard_normal((L, 2, 4)), rng.standard_normal((L, 1, 4)), rng.standard_normal((L, 1, 4))
    O, LSE = oracle.ring_forward(q, k, v, R, layout=layout, offsets=docs, chunks_per_rank=m)
    pos = oracle.ring_positions(L, R, layout, docs, m)
    Of, Lf = oracle.attention(q, k, v, offsets=docs)
    np.testing.assert_allclose(oracle.unshard(O.reshape(L, 2, 4), pos), Of, rtol=1e-10, atol=1e-12)
    lse_global = np.empty_like(Lf)
    lse_global[:, pos] = LSE.transpose(1, 0, 2).reshape(2, L)
    np.testing.assert_allclose(lse_global, Lf, rtol=1e-10, atol=1e-12)


@SETTINGS
@given(ring_plans())
def test_index_maps_are_permutations(plan):
    L, R, layout, m, docs, _ = plan
    pos = oracle.ring_positions(L, R, layout, docs, m)
    assert sorted(pos.tolist()) == list(range(L))


@st.composite
def tile_plans(draw):
    R = draw(st.integers(1, 3))
    U = draw(st.sampled_from([1, 2]))
    layout = draw(st.sampled_from([0, 1, 2]))
    m = {0: 1, 1: 2, 2: 2}[layout]
    chunk = draw(st.sampled_from([64, 128, 200, 256, 300]))
    L = R * m * chunk
    cuts = sorted(draw(st.sets(st.integers(1, L - 1), max_size=3)))
    docs = [0] + cuts + [L] if cuts else None
    return L, R, U, layout, m, docs, draw(st.booleans()), draw(st.booleans())


@settings(max_examples=15, deadline=None, derandomize=True)
@given(tile_plans())
def test_touched_tiles_hold_every_visible_pair_once(plan):
    L, R, U, layout, m, docs, allgather, per_step = plan
    t = tile_classes(L, R, U, layout, docs, m, allgather=allgather, per_step=per_step and not allgather)
    pos = oracle.ring_positions(L, R, layout, docs, m)
    T = L // R
    got = np.zeros(R * U, dtype=np.int64)
    for (a, q0, ln, s), rows in t.items():
        r = a // U
        for k0, klen, c0, c1 in rows:
            for i, c in enumerate((c0, c1)):
                qp = pos[r * T + q0 + i * 128: r * T + q0 + min(ln, (i + 1) * 128)]
                vis = int(oracle.visible(qp, np.arange(k0, k0 + klen), docs).sum()) if len(qp) else 0
                if c == 0:
                    assert vis == 0
                else:
                    got[a] += vis
                    if c == 2:
                        assert vis == len(qp) * 128
    want = np.repeat(oracle.rank_visible_pairs(L, R, layout, docs, m), U)
    np.testing.assert_array_equal(got, want)


def test_log_sum_exp_reference_value():
    # Sanity of the helper arithmetic the properties lean on: ln(e^1 + e^2).
    o, l = oracle.merge([(np.ones((1, 1, 1)), np.full((1, 1), 1.0)), (np.zeros((1, 1, 1)), np.full((1, 1), 2.0))])
    assert math.isclose(l.item(), math.log(math.e + math.e ** 2), rel_tol=1e-14)
    assert math.isclose(o.item(), math.e / (math.e + math.e ** 2), rel_tol=1e-14)
