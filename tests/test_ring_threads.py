"""The ring exchange run as one host thread per rank (oracle.ring_threads):
it reproduces the single-loop ring forward bit for bit, a late chunk within
the limit changes nothing, and a dropped chunk, a dead rank or a duplicated
message end the whole ring with a clear per-rank status within about one
wait limit -- failure detection with the failure made on the host."""
import time

import numpy as np
import pytest

import oracle
from oracle.ring_threads import RingFailure, ring_forward_threads


def _inputs(L, Hq, Hkv, d, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((L, Hq, d)), rng.standard_normal((L, Hkv, d)), rng.standard_normal((L, Hkv, d)))


@pytest.mark.parametrize("R,layout,docs", [(4, 1, None), (3, 0, [0, 20, 50, 96]), (4, 2, [0, 33, 128]),
                                           (1, 0, None)])
def test_threads_equal_single_loop_ring(R, layout, docs):
    q, k, v = _inputs(128 if R != 3 else 96, 4, 2, 16, 7)
    O, LSE = ring_forward_threads(q, k, v, R, layout=layout, offsets=docs, chunks_per_rank=2)
    O_ref, LSE_ref = oracle.ring_forward(q, k, v, R, layout=layout, offsets=docs, chunks_per_rank=2)
    assert np.array_equal(O, O_ref) and np.array_equal(LSE, LSE_ref)
    # ... and, unsharded, the full attention.
    pos = oracle.ring_positions(q.shape[0], R, layout, docs, 2)
    Of, Lf = oracle.attention(q, k, v, offsets=docs)
    assert np.abs(oracle.unshard(O.reshape(-1, *O.shape[2:]), pos) - Of).max() < 1e-12
    assert np.abs(LSE.transpose(1, 0, 2).reshape(LSE.shape[1], -1)[:, np.argsort(pos)] - Lf).max() < 1e-12


def test_late_chunk_within_limit_changes_nothing():
    q, k, v = _inputs(128, 2, 2, 16, 3)
    ref = oracle.ring_forward(q, k, v, 4, layout=1)
    O, LSE = ring_forward_threads(q, k, v, 4, layout=1, timeout=2.0, delay=(1, 0, 0.3))
    assert np.array_equal(O, ref[0]) and np.array_equal(LSE, ref[1])


@pytest.mark.parametrize("R,rank,step", [(4, 1, 0), (4, 3, 2), (2, 0, 0)])
def test_dropped_chunk_times_out_and_aborts_the_ring(R, rank, step):
    q, k, v = _inputs(64 * R, 2, 1, 16, 5)
    limit = 0.4
    t0 = time.monotonic()
    with pytest.raises(RingFailure) as ei:
        ring_forward_threads(q, k, v, R, layout=1, timeout=limit, drop=(rank, step))
    elapsed = time.monotonic() - t0
    st = ei.value.status
    recv = (rank + 1) % R
    # The receiver notices the gap: by its limit, or earlier when the sender
    # goes on and its next step's chunk arrives in place of the lost one.
    assert st[recv] in (f"timeout at step {step + 1} waiting for rank {rank}",
                        f"protocol: expected (rank {rank}, step {step}), got ({rank}, {step + 1})"), st
    assert all(s in ("aborted", "ok") for r, s in enumerate(st) if r != recv), st
    # The others left on the abort, not on their own limits.
    assert elapsed < limit + 5.0, elapsed


def test_late_chunk_past_limit_is_a_timeout():
    q, k, v = _inputs(128, 2, 1, 16, 5)
    with pytest.raises(RingFailure) as ei:
        ring_forward_threads(q, k, v, 4, layout=1, timeout=0.2, delay=(2, 1, 1.0))
    assert ei.value.status[3].startswith("timeout at step 2"), ei.value.status


def test_dead_rank_is_reported_and_others_abort():
    q, k, v = _inputs(128, 2, 1, 16, 9)
    with pytest.raises(RingFailure) as ei:
        ring_forward_threads(q, k, v, 4, layout=0, timeout=5.0, die=(2, 1))
    st = ei.value.status
    assert st[2] == "error: injected failure at step 1", st
    assert all(s in ("aborted", "ok", ) or s.startswith("timeout") for r, s in enumerate(st) if r != 2), st


@pytest.mark.parametrize("step", [0, 2])
def test_duplicate_message_is_a_protocol_error(step):
    q, k, v = _inputs(128, 2, 1, 16, 11)
    with pytest.raises(RingFailure) as ei:
        ring_forward_threads(q, k, v, 4, layout=1, timeout=1.0, duplicate=(0, step))
    assert ei.value.status[1].startswith("protocol"), ei.value.status
