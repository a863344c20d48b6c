"""The forward kernel's tile choices, exported by cp_tile_classes (the same
device functions the attention kernel runs), equal the classes oracle.tiles
derives from the mask alone, entry by entry: the same query blocks, the same
key tiles, and for each query tile the same decision to skip the tile, mask
it, or take it whole.  A single ring step (emit-partials) is walked in the
oracle's order; a launch over all ring steps visits the chunks in position
order (the oracle lists them in ring order), so there the tiles of each
query block are compared sorted by key position."""
import os
import sys

import pytest
import torch

sys.path.insert(0, os.path.dirname(__file__))

pytestmark = pytest.mark.gpu

from oracle.tiles import tile_classes  # noqa: E402


@pytest.fixture(scope="module")
def cpa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import context_long_sequence_gb300 as m
    return m


CASES = [  # id, L, R, U, layout, docs, chunks_per_rank, allgather, emit_partials
    ("contig_R1", 1280, 1, 1, 0, None, 4, False, False),
    ("zigzag_R4_docs", 2048, 4, 1, 1, [0, 100, 333, 1500, 2048], 4, False, False),
    ("zigzag_R3_ragged_chunks", 1440, 3, 1, 1, [0, 250, 1440], 4, False, False),
    ("ulysses_U2_R2", 2048, 2, 2, 1, [0, 900, 2048], 4, False, False),
    ("balanced_R4_m4", 4096, 4, 1, 2, [0, 50, 1200, 3000, 4096], 4, False, False),
    ("allgather_R4", 2048, 4, 1, 1, [0, 700, 2048], 4, True, False),
    ("allgather_balanced", 1536, 3, 1, 2, [0, 200, 1100, 1536], 4, True, False),
    ("partials_R4", 2048, 4, 1, 1, [0, 1000, 2048], 4, False, True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_tile_classes_match_oracle(cpa, case):
    _, L, R, U, layout, docs, m, ag, ep = case
    plan = cpa.Plan(L, 4, 2, 128, ulysses_degree=U, ring_degree=R, layout=layout, doc_offsets=docs,
                    chunks_per_rank=m, kv_exchange=cpa.CP_KV_ALLGATHER if ag else cpa.CP_KV_RING,
                    emit_partials=ep)
    rows = cpa.cp_tile_classes(plan)
    got = {}
    order = []
    for a, q0, ln, step, k0, klen, c0, c1 in rows.tolist():
        key = (a, q0, ln, step)
        if key not in got:
            got[key] = []
            order.append(key)
        elif order[-1] != key:
            raise AssertionError(f"rows of item {key} are not contiguous")
        got[key].append((k0, klen, c0, c1))
    want = tile_classes(L, R, U, layout, docs, m, allgather=ag, per_step=ep)
    # An item the kernel walks with no tile at all (nothing visible) has no rows.
    want = {k: v for k, v in want.items() if v}
    assert set(got) == set(want), (sorted(set(got) ^ set(want))[:10])
    for k in want:
        step = k[3]
        if step < 0 and R > 1 and not ag:
            assert sorted(got[k]) == sorted(want[k]), (k, got[k], want[k])
            kpos = [t[0] for t in got[k]]
            assert kpos == sorted(kpos), (k, "fused walk not in position order", kpos)
        else:
            assert got[k] == want[k], (k, got[k], want[k])
