"""Work-balanced sharding for packed documents (CPU): the per-rank work
spread (max over ranks / mean of the visible pairs whose query a rank holds)
of the balanced layout against zigzag, on the packed-document workload's
seeded documents (L = 131072, R = 16)."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(__file__))

import oracle  # noqa: E402
import workloads  # noqa: E402


def _spread(work):
    work = np.asarray(work, dtype=np.float64)
    return work.max() / work.mean()


def test_balanced_spread_beats_zigzag_on_packed_documents():
    w = workloads.WORKLOADS[3]
    offs = workloads.workload_doc_offsets(w)
    zig = _spread(oracle.rank_visible_pairs(w.L, w.ring, oracle.LAYOUT_ZIGZAG, offs))
    bal = {m: _spread(oracle.rank_visible_pairs(w.L, w.ring, oracle.LAYOUT_BALANCED, offs, m)) for m in (4, 8)}
    # Zigzag balances causal work only within one document: with ~24 packed
    # documents the busiest rank does about 2.5x the mean work.
    assert zig > 2.0
    assert bal[4] < 1.1 and bal[8] < 1.01
    assert bal[8] <= bal[4] < zig


def test_balanced_equals_zigzag_without_documents():
    for L, R in [(131072, 16), (65536, 8)]:
        assert np.array_equal(oracle.ring_positions(L, R, oracle.LAYOUT_BALANCED, None, 2),
                              oracle.ring_positions(L, R, oracle.LAYOUT_ZIGZAG))
