"""Tile classes of the blocked causal forward, from the mask alone.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle``): only the tests may
import it; the CUDA path never calls it.

A blocked attention forward processes a query block against key tiles and
can skip a tile no query row of the block can see, and skip the mask for a
tile every row sees whole.  This module states, from the visibility mask
M(i,k) of ``oracle.attention.visible`` and nothing else, which key tiles a
query block has to touch and how, so that the device's choices can be
compared with it entry by entry (the debug table ``cp_tile_classes``):

* query blocks: per attention rank, per contiguous-position chunk of its
  slots, blocks of 256 slots from the chunk start (the last one ragged),
  each split into query tiles 0 and 1 of up to 128 rows; with per-step
  partials, one block per ring step;
* key tiles, in ring order ([MTX] nougat.kr, "MaxText long-context training
  and KV parallelism", section "Split heads or rotate KV": at step s the
  chunk of ring rank (r - s) mod R): that rank's chunks in slot order, 128
  slots from each chunk's start; with all-gathered K/V ([MTX] "Why KV comes
  back together"), 128-position tiles of the whole sequence;
* class of a key tile for a query tile: 0 if no row of the query tile sees
  any of its keys, 2 if every row sees every key and the tile has 128 keys
  (a shorter tile still needs its missing columns masked), 1 otherwise;
* a block lists the key tiles some row of it sees (class 0 for both query
  tiles means the tile is not touched at all), in the order above.
"""
from __future__ import annotations

import numpy as np

from .attention import LAYOUT_BALANCED, LAYOUT_CONTIGUOUS, LAYOUT_ZIGZAG, ring_positions, visible

TILE = 128
BLOCK = 256


def chunks_of(layout: int, chunks_per_rank: int) -> int:
    return {LAYOUT_CONTIGUOUS: 1, LAYOUT_ZIGZAG: 2, LAYOUT_BALANCED: chunks_per_rank}[layout]


def _class(vis: np.ndarray, klen: int) -> int:
    if vis.size == 0 or not vis.any():
        return 0
    return 2 if (vis.all() and klen == TILE) else 1


def tile_classes(L, R, U=1, layout=LAYOUT_CONTIGUOUS, offsets=None, chunks_per_rank=4, allgather=False,
                 per_step=False):
    """{(a, q0, len, step): [(kpos0, klen, class0, class1), ...]} for every
    query block of the plan (step = -1 when a block covers all ring steps)."""
    T = L // R
    m = chunks_of(layout, chunks_per_rank)
    chunk = T // m
    pos = ring_positions(L, R, layout, offsets, chunks_per_rank)
    out = {}
    for a in range(R * U):
        r = a // U
        for c in range(m):
            for t0 in range(0, chunk, BLOCK):
                q0 = c * chunk + t0
                ln = min(BLOCK, chunk - t0)
                qpos = [pos[r * T + q0 + t * TILE: r * T + q0 + min(ln, (t + 1) * TILE)] for t in (0, 1)]
                for steps in ([[s] for s in range(R)] if per_step else [list(range(R))]):
                    key_tiles = []
                    if allgather:
                        key_tiles = [np.arange(k0, min(L, k0 + TILE)) for k0 in range(0, L, TILE)]
                    else:
                        for s in steps:
                            src = (r - s) % R
                            for cc in range(m):
                                for k0 in range(0, chunk, TILE):
                                    sl = src * T + cc * chunk + k0
                                    key_tiles.append(pos[sl: sl + min(TILE, chunk - k0)])
                    rows = []
                    for kp in key_tiles:
                        cls = [_class(visible(qp, kp, offsets), len(kp)) for qp in qpos]
                        if cls[0] or cls[1]:
                            rows.append((int(kp[0]), len(kp), cls[0], cls[1]))
                    out[(a, q0, ln, steps[0] if per_step else -1)] = rows
    return out
