"""Pins of oracle.tiles (the tile classes of the blocked forward, from the
mask alone) and planted mistakes that the pins must catch.

Pins: hand-worked tables (tests/golden/tile_classes_examples.json); a closed
form for one rank without documents; coverage -- over every query block, the
visible (query, key) pairs inside the touched tiles add up to each rank's
visible pairs, so no tile that holds a visible pair is left out and none is
listed twice; the ring order of the key tiles; all-gathered K/V giving the
same tiles as the ring when the tile grids coincide; a ragged key tile is
never wholly visible."""
import json
import os
import types

import numpy as np
import pytest

import oracle
import oracle.tiles as tiles_mod

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = json.load(open(os.path.join(HERE, "golden", "tile_classes_examples.json")))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "tiles.py")


def pin_golden(tm):
    for c in GOLDEN["cases"]:
        t = tm.tile_classes(c["L"], c["R"], 1, c["layout"], c["offsets"])
        want = {tuple(int(x) for x in k.split(",")): [tuple(r) for r in v] for k, v in c["blocks"].items()}
        assert set(t) == set(want), (sorted(t), sorted(want))
        for k, v in want.items():
            assert [tuple(r) for r in t[k]] == v, (k, t[k], v)


def pin_closed_form(tm):
    L = 1280
    t = tm.tile_classes(L, 1)
    assert sorted(t) == [(0, q, min(256, L - q), -1) for q in range(0, L, 256)]
    for (a, q, ln, s), rows in t.items():
        want = []
        for k0 in range(0, L, 128):
            cls = []
            for qt in (q, q + 128):
                if qt >= q + ln or k0 > qt + 127:
                    cls.append(0)
                elif k0 + 127 <= qt:
                    cls.append(2)
                else:
                    cls.append(1)
            if cls[0] or cls[1]:
                want.append((k0, 128, cls[0], cls[1]))
        assert [tuple(r) for r in rows] == want, (q, rows, want)


PLANS = [  # L, R, U, layout, offsets, chunks_per_rank, allgather, per_step
    (768, 3, 1, 1, None, 4, False, False),
    (1024, 4, 1, 1, [0, 100, 333, 700, 1024], 4, False, False),
    (1024, 2, 2, 2, [0, 450, 1024], 4, False, False),
    (960, 2, 1, 1, [0, 17, 960], 4, False, True),
    (1024, 4, 1, 0, [0, 600, 1024], 4, True, False),
    (1536, 3, 1, 2, [0, 200, 1100, 1536], 4, True, False),
]


def _tile_pairs(qpos, k0, klen, offsets):
    return int(oracle.visible(qpos, np.arange(k0, k0 + klen), offsets).sum())


def pin_coverage(tm):
    for L, R, U, layout, docs, m, ag, ps in PLANS:
        t = tm.tile_classes(L, R, U, layout, docs, m, allgather=ag, per_step=ps)
        pos = oracle.ring_positions(L, R, layout, docs, m)
        T = L // R
        per_rank = np.zeros(R * U, dtype=np.int64)
        for (a, q0, ln, s), rows in t.items():
            r = a // U
            qp = [pos[r * T + q0 + i * 128: r * T + q0 + min(ln, (i + 1) * 128)] for i in (0, 1)]
            for k0, klen, c0, c1 in rows:
                for i, c in enumerate((c0, c1)):
                    if c:
                        per_rank[a] += _tile_pairs(qp[i], k0, klen, docs)
        want = np.repeat(oracle.rank_visible_pairs(L, R, layout, docs, m), U)
        assert np.array_equal(per_rank, want), (L, R, U, layout, per_rank, want)


def pin_ring_order(tm):
    for L, R, U, layout, docs, m, ag, ps in PLANS:
        if ag or ps:
            continue
        pos = oracle.ring_positions(L, R, layout, docs, m)
        owner = np.empty(L, dtype=np.int64)
        owner[pos] = np.arange(L) // (L // R)
        for (a, q0, ln, s), rows in tm.tile_classes(L, R, U, layout, docs, m).items():
            r = a // U
            steps = [(r - owner[k0]) % R for k0, _, _, _ in rows]
            assert steps == sorted(steps), (a, q0, steps)


def pin_allgather_matches_ring_grid(tm):
    L, R, docs = 1024, 4, [0, 300, 1024]   # contiguous, 256 slots per rank: the two tile grids coincide
    ring = tm.tile_classes(L, R, 1, 0, docs)
    ag = tm.tile_classes(L, R, 1, 0, docs, allgather=True)
    assert set(ring) == set(ag)
    for k in ring:
        assert sorted(ring[k]) == sorted(ag[k]), k


def pin_ragged_tile_never_full(tm):
    t = tm.tile_classes(960, 2, 1, 1, None)      # chunks of 240 slots: tiles of 128 and 112 keys
    pos = oracle.ring_positions(960, 2, 1)
    seen_all_visible_ragged = False
    for (a, q0, ln, s), rows in t.items():
        qp = pos[a * 480 + q0: a * 480 + q0 + min(ln, 128)]
        for k0, klen, c0, _ in rows:
            if klen != 128:
                assert c0 != 2 and _ != 2
                if c0 and _tile_pairs(qp, k0, klen, None) == len(qp) * klen:
                    seen_all_visible_ragged = True
    assert seen_all_visible_ragged


PINS = [pin_golden, pin_closed_form, pin_coverage, pin_ring_order, pin_allgather_matches_ring_grid,
        pin_ragged_tile_never_full]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(tiles_mod)


MUTATIONS = {
    "ring_order_reversed": ("src = (r - s) % R", "src = (r + s) % R"),
    "full_ignores_klen": ("vis.all() and klen == TILE", "vis.all()"),
    "full_if_any_row": ("2 if (vis.all() and klen == TILE)", "2 if (vis.any() and klen == TILE)"),
    "key_slot_drops_chunk": ("sl = src * T + cc * chunk + k0", "sl = src * T + k0"),
    "block_of_128": ("BLOCK = 256", "BLOCK = 128"),
    "allgather_first_tile_dropped": ("range(0, L, TILE)", "range(TILE, L, TILE)"),
    "per_step_one_source": ("[[s] for s in range(R)]", "[[0] for s in range(R)]"),
    "query_tile_offset": ("pos[r * T + q0 + t * TILE:", "pos[r * T + t * TILE:"),
}


def _mutant(old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    src = src.replace(old, new).replace("from .attention import", "from oracle.attention import")
    mod = types.ModuleType("tiles_mutant")
    exec(compile(src, "tiles_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name):
    mod = _mutant(*MUTATIONS[name])
    failed = []
    for pin in PINS:
        try:
            pin(mod)
        except Exception:
            failed.append(pin.__name__)
    assert failed, f"no pin catches mutation {name}"
