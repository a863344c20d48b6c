"""Ring (P2P) exchange protocol emulated with one host thread per rank.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle``): only the tests may
import it; the CUDA path never calls it.

[MTX] nougat.kr, "MaxText long-context training and KV parallelism", section
"Split heads or rotate KV": with P2P each chip keeps its own queries, computes
a partial with the K/V chunk it holds, passes the chunk to the next chip and
merges the partials.  ``ring_forward`` in ``oracle.attention`` evaluates the
same partials in one loop; this module runs the exchange itself, so that the
tests can check the protocol (order of arrival, tags, termination) and inject
the faults the pages list for long runs ([L3P] siliconandsystems.com, "Llama
3 parallelism", section "Long context changes more than attention cost":
slow ranks and failures) on the host, without a GPU:

* rank r holds the chunk of rank (r - s) mod R at step s, computes its
  partial, folds it into its running (O, LSE) with ``merge_pair`` (the same
  fold, in the same order, as ``merge``), and, unless s is the last step,
  sends the chunk to rank (r + 1) mod R and waits for the one from rank
  (r - 1) mod R;
* every wait is bounded: a receiver that gets nothing within ``timeout``
  seconds fails with a timeout and raises the shared abort event; every other
  rank polls that event while it waits and leaves ("aborted") instead of
  waiting out its own limit, so a lost chunk ends the whole ring within about
  one ``timeout`` -- the host-side analogue of the kernels' bounded waits and
  CTA abort flag;
* a message carries (source rank, step); a receiver that gets another one
  than it expects fails with a protocol error.

Faults (all injected on the host): ``drop=(rank, step)`` -- that rank does not
send at that step; ``delay=(rank, step, seconds)`` -- it sends late;
``die=(rank, step)`` -- it raises before computing that step;
``duplicate=(rank, step)`` -- it sends the step's chunk twice.
"""
from __future__ import annotations

import queue
import threading
import time

import numpy as np

from .attention import LAYOUT_CONTIGUOUS, attention_rows, merge_pair, ring_positions, shard


class RingFailure(RuntimeError):
    """The ring did not complete.  ``status[r]`` says what became of rank r:
    "ok", "timeout ...", "aborted", "error ...", "protocol ..."."""

    def __init__(self, status):
        self.status = status
        super().__init__("ring failed: " + "; ".join(f"rank {r}: {s}" for r, s in enumerate(status)))


_POLL_S = 0.005


def _recv(inbox: "queue.Queue", abort: threading.Event, timeout: float):
    """Bounded wait for one message; None on timeout, "abort" if another rank failed."""
    t_end = time.monotonic() + timeout
    while True:
        if abort.is_set():
            return "abort"
        left = t_end - time.monotonic()
        if left <= 0:
            return None
        try:
            return inbox.get(timeout=min(_POLL_S, left))
        except queue.Empty:
            continue


def ring_forward_threads(q, k, v, R, layout=LAYOUT_CONTIGUOUS, offsets=None, causal=True, scale=None,
                         chunks_per_rank=4, timeout=2.0, drop=None, delay=None, die=None, duplicate=None):
    """Ring forward with one thread per rank; returns (O [R][n][Hq][d], LSE
    [R][Hq][n]) in slot order, like ``ring_forward``, or raises RingFailure.

    Inputs are global-order [L][H][d] arrays (fp64 or exactly representable).
    """
    L = q.shape[0]
    n = L // R
    pos = ring_positions(L, R, layout, offsets, chunks_per_rank)
    qs, ks, vs = shard(q, pos), shard(k, pos), shard(v, pos)
    inbox = [queue.Queue() for _ in range(R)]
    abort = threading.Event()
    status = ["ok"] * R
    out = [None] * R

    def rank_main(r):
        try:
            q_r = qs[r * n:(r + 1) * n]
            q_pos = pos[r * n:(r + 1) * n]
            held = (r, ks[r * n:(r + 1) * n], vs[r * n:(r + 1) * n], pos[r * n:(r + 1) * n])
            o = lse = None
            for s in range(R):
                if die is not None and die == (r, s):
                    raise RuntimeError(f"injected failure at step {s}")
                src, k_c, v_c, k_pos = held
                part = attention_rows(q_r, k_c, v_c, q_pos=q_pos, k_pos=k_pos, offsets=offsets,
                                      causal=causal, scale=scale)
                o, lse = part if s == 0 else merge_pair(o, lse, *part)
                if s == R - 1:
                    break
                # Pass the held chunk on, then take the next one.
                if delay is not None and delay[:2] == (r, s):
                    time.sleep(delay[2])
                if drop is None or drop != (r, s):
                    inbox[(r + 1) % R].put((r, s, held))
                    if duplicate is not None and duplicate == (r, s):
                        inbox[(r + 1) % R].put((r, s, held))
                msg = _recv(inbox[r], abort, timeout)
                if msg == "abort":
                    status[r] = "aborted"
                    return
                if msg is None:
                    status[r] = f"timeout at step {s + 1} waiting for rank {(r - 1) % R}"
                    abort.set()
                    return
                m_src, m_step, chunk = msg
                if m_src != (r - 1) % R or m_step != s:
                    status[r] = f"protocol: expected (rank {(r - 1) % R}, step {s}), got ({m_src}, {m_step})"
                    abort.set()
                    return
                if chunk[0] != (r - s - 1) % R:
                    status[r] = f"protocol: step {s + 1} brought the chunk of rank {chunk[0]}"
                    abort.set()
                    return
                held = chunk
            # Nothing may be left over: an extra message is a protocol error.
            if not inbox[r].empty():
                status[r] = "protocol: unexpected extra message"
                abort.set()
                return
            out[r] = (o, lse)
        except Exception as e:  # noqa: BLE001 -- the failure is the rank's status
            status[r] = f"error: {e}"
            abort.set()

    threads = [threading.Thread(target=rank_main, args=(r,), daemon=True) for r in range(R)]
    for t in threads:
        t.start()
    # Every wait inside is bounded, so each thread ends within about R
    # computations plus one timeout; the join limit is a second fence.
    for t in threads:
        t.join(timeout=60.0 + R * timeout)
    if any(t.is_alive() for t in threads):
        abort.set()
        raise RingFailure([s if not t.is_alive() else "hung" for s, t in zip(status, threads)])
    # An extra message can arrive after its receiver finished: check again.
    for r in range(R):
        if status[r] == "ok" and not inbox[r].empty():
            status[r] = "protocol: unexpected extra message"
    if any(s != "ok" for s in status):
        raise RingFailure(status)
    return np.stack([o for o, _ in out]), np.stack([lse for _, lse in out])
