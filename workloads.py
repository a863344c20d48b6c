"""Seeded synthetic inputs for context-parallel causal attention.

This module is shared by the oracle's tests, the GPU parity tests and the
benchmark.  It holds the five workload shapes and the random-number recipes
only: no attention, merge or reshard arithmetic lives here, so that the CPU
oracle and the CUDA path stay independent of each other.

Recipes (stated once, used everywhere):

* Q, K, V (and dO for the backward) are drawn as float32 ``randn`` in that
  order from one ``torch.Generator`` seeded with ``1000 + config index`` and
  rounded to bfloat16 (round-to-nearest-even, torch's ``.to(bfloat16)``).
* "K scaled by 0.5" multiplies the bf16 K by 0.5, which is exact in bf16.
* Packed-document lengths are lognormal(mu=ln 4096, sigma=1) draws from
  ``numpy.random.default_rng(seed)``, rounded half-to-even, clipped to
  [256, 32768], drawn until their sum reaches L, and the last one trimmed so
  the lengths sum to exactly L (the last may fall below 256).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

LAYOUT_CONTIGUOUS = 0
LAYOUT_ZIGZAG = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    L: int
    Hq: int
    Hkv: int
    d: int
    ulysses: int          # U, Ulysses (all-to-all) degree
    ring: int             # R, ring (P2P) degree
    layout: int           # LAYOUT_CONTIGUOUS or LAYOUT_ZIGZAG
    docs: bool            # packed-document (block-causal) mask
    backward: bool        # the workload includes dQ, dK, dV
    emit_partials: bool   # forward writes per-ring-step partials, merged afterwards
    k_scale: float = 1.0  # K multiplied by this after bf16 rounding
    seed: int = 0

    @property
    def P(self) -> int:
        return self.ulysses * self.ring


# The five workloads, in order.  Index i uses seed 1000 + i.
WORKLOADS = [
    Workload("ring_fwd_L1K_P4", 1024, 4, 4, 64, 1, 4, LAYOUT_CONTIGUOUS,
             docs=False, backward=False, emit_partials=True, seed=1000),
    Workload("ulysses_fwd_L16K_U4", 16384, 32, 8, 128, 4, 1, LAYOUT_CONTIGUOUS,
             docs=False, backward=False, emit_partials=False, seed=1001),
    Workload("ring_fwdbwd_L64K_R8_zigzag", 65536, 32, 8, 128, 1, 8, LAYOUT_ZIGZAG,
             docs=False, backward=True, emit_partials=False, k_scale=0.5, seed=1002),
    Workload("docs_ring_fwd_L128K_R16", 131072, 32, 8, 128, 1, 16, LAYOUT_ZIGZAG,
             docs=True, backward=False, emit_partials=False, seed=1003),
    Workload("usp_fwd_L1M_U4xR8_zigzag", 1048576, 32, 8, 128, 4, 8, LAYOUT_ZIGZAG,
             docs=False, backward=False, emit_partials=False, seed=1004),
]

WORKLOAD_BY_NAME = {w.name: w for w in WORKLOADS}


def doc_lengths(L: int, seed: int, mu: float = math.log(4096.0), sigma: float = 1.0,
                lo: int = 256, hi: int = 32768) -> np.ndarray:
    """Seeded packed-document lengths summing to exactly L (recipe above)."""
    rng = np.random.default_rng(seed)
    out = []
    total = 0
    while total < L:
        n = int(np.clip(np.rint(rng.lognormal(mu, sigma)), lo, hi))
        out.append(n)
        total += n
    out[-1] -= total - L
    if out[-1] <= 0:  # cannot happen with lo >= 1, kept as a guard
        out.pop()
    return np.asarray(out, dtype=np.int64)


def doc_offsets(lengths: np.ndarray) -> np.ndarray:
    """Offsets [0, l0, l0+l1, ..., L] of packed documents, int32."""
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def randn_bf16(gen: torch.Generator, shape, device) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_inputs(L: int, Hq: int, Hkv: int, d: int, seed: int, device="cpu",
                k_scale: float = 1.0, with_do: bool = False):
    """Global-order Q [L,Hq,d], K, V [L,Hkv,d] (and dO [L,Hq,d]) in bf16.

    Draw order is Q, K, V, dO from one generator seeded with ``seed``.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q = randn_bf16(gen, (L, Hq, d), device)
    k = randn_bf16(gen, (L, Hkv, d), device)
    v = randn_bf16(gen, (L, Hkv, d), device)
    if k_scale != 1.0:
        k = k * k_scale
    out = {"q": q, "k": k, "v": v}
    if with_do:
        out["do"] = randn_bf16(gen, (L, Hq, d), device)
    return out


def workload_inputs(w: Workload, device="cpu"):
    return make_inputs(w.L, w.Hq, w.Hkv, w.d, w.seed, device=device,
                       k_scale=w.k_scale, with_do=w.backward)


def workload_doc_offsets(w: Workload):
    if not w.docs:
        return None
    return doc_offsets(doc_lengths(w.L, w.seed))


def sample_rows(L: int, boundaries, per_head: int, seed: int) -> np.ndarray:
    """Sorted unique global positions to check at large L: the first and last
    position of every segment delimited by ``boundaries`` (chunk and document
    starts) plus ``per_head`` seeded random positions."""
    rng = np.random.default_rng(seed)
    b = sorted(set(int(x) for x in boundaries) | {0, L})
    pts = set()
    for s, e in zip(b[:-1], b[1:]):
        if e > s:
            pts.add(s)
            pts.add(e - 1)
    pts.update(int(x) for x in rng.integers(0, L, size=per_head))
    return np.asarray(sorted(pts), dtype=np.int64)
