"""Ring transport of K/V chunks between processes (one process per GPU).

The pages' ring (P2P) context parallelism keeps each rank's queries in
place and passes the K/V chunks around the ring: every rank computes a
partial result with the chunk it holds, sends that chunk on to the next
rank, receives the next one from the previous rank while it computes, and
merges the partials ([MTX] nougat.kr "MaxText long-context training and KV
parallelism", section "Split heads or rotate KV"; USP = Ulysses all-to-all
groups x ring).  In the backward the chunk's dK and dV travel with it and
arrive back at the owner after the last step.

This module is the host side of that exchange.  It owns the schedule:
which chunk each rank holds at each step, which buffer the next chunk lands
in (one spare buffer per process: receive into the spare while computing on
the others, then rotate), the message tags, the bounded waits, and the
abort that one failing rank raises for all the others through the
process group's store.  The arithmetic of each step is done by a `kernels`
object: `CudaRingKernels` below calls the library's per-step entry points
(cp_attn_fwd_step, cp_attn_bwd_delta, cp_attn_bwd_step, cp_merge_lse) on the
current CUDA stream; tests may pass another implementation.

Placement: N processes, ring degree R with N | R.  Process p holds ring
ranks [p*R/N, (p+1)*R/N) with all U of their Ulysses members (attention
rank a = r*U + u), so the Ulysses exchange stays inside a process (the
library's reshard kernel) and only the ring crosses processes.  A chunk is
one ring rank's K and V for all U members, two [U][T][Hkv/U][d] tensors
sent as two messages (in the backward also its fp32 dK and dV).

Point-to-point uses torch.distributed isend/irecv (NCCL between GPUs, gloo
on CPU): plain sends into local buffers, no peer memory access by any
kernel.  On GPUs, ProcessGroupNCCL orders each send or receive after the
work already queued on the current stream and `wait` makes the current
stream wait for it, so the transfers overlap the step's kernels.
"""
from __future__ import annotations

import datetime
from dataclasses import dataclass

import torch

ABORT_KEY = "cp_ring_abort"
TAG_KV = 0          # tags: kind * 1_000_000 + step (gloo matches on tags; NCCL ignores them)
TAG_GRAD = 1


class TransportError(RuntimeError):
    """A ring exchange did not complete: `kind` is 'timeout' (a wait ran
    past its limit), 'peer_abort' (another rank aborted first) or 'error'
    (the communication call failed); `step` and `peer` say where."""

    def __init__(self, kind: str, rank: int, step: int, peer: int, detail: str = ""):
        self.kind, self.rank, self.step, self.peer, self.detail = kind, rank, step, peer, detail
        super().__init__(f"ring transport {kind} on process {rank} at step {step} (peer {peer}): {detail}")


class DistComm:
    """Point-to-point over an initialised torch.distributed process group,
    with a bounded wait on every transfer and an abort flag in the group's
    store that every process checks before each step."""

    def __init__(self, timeout_s: float = 60.0):
        import torch.distributed as dist
        self.dist = dist
        self.rank = dist.get_rank()
        self.world = dist.get_world_size()
        self.timeout = datetime.timedelta(seconds=timeout_s)
        self.store = dist.distributed_c10d._get_default_store()

    def isend(self, t: torch.Tensor, peer: int, tag: int):
        return self.dist.isend(t, dst=peer, tag=tag)

    def irecv(self, t: torch.Tensor, peer: int, tag: int):
        return self.dist.irecv(t, src=peer, tag=tag)

    def wait(self, handle, step: int, peer: int):
        try:
            handle.wait(timeout=self.timeout)
        except Exception as e:  # the backend's timeout or a failed peer
            kind = "timeout" if "imed out" in str(e) or "imeout" in str(e) else "error"
            self.abort(f"{kind} on process {self.rank} at step {step}")
            raise TransportError(kind, self.rank, step, peer, str(e)[:200]) from e

    def check_abort(self, step: int):
        if self.store.check([ABORT_KEY]):
            raise TransportError("peer_abort", self.rank, step, -1, self.store.get(ABORT_KEY).decode())

    def abort(self, why: str):
        try:
            self.store.set(ABORT_KEY, why)
        except Exception:
            pass


class LocalComm:
    """One process holding the whole ring: a send to itself is kept and the
    matching receive copies it (stream-ordered on the current stream)."""

    rank, world = 0, 1

    def __init__(self):
        self._sent = {}

    def isend(self, t, peer, tag):
        self._sent[tag] = t
        return None

    def irecv(self, t, peer, tag):
        t.copy_(self._sent.pop(tag))
        return None

    def wait(self, handle, step, peer):
        return None

    def check_abort(self, step):
        return None

    def abort(self, why):
        return None


@dataclass
class RingPlacement:
    """Which ring ranks this process holds: [r0, r0 + Rl)."""
    R: int
    U: int
    world: int
    rank: int

    def __post_init__(self):
        if self.R % self.world:
            raise ValueError(f"ring degree {self.R} is not a multiple of the process count {self.world}")
        self.Rl = self.R // self.world
        self.r0 = self.rank * self.Rl
        self.next = (self.rank + 1) % self.world
        self.prev = (self.rank - 1) % self.world


def _post(comm, place: RingPlacement, last, spare, step: int, tag_kind: int):
    """Send the tensors of `last` (the chunk of this process's last ring
    rank) to the next process and receive the previous process's into
    `spare`; returns the handles."""
    hs, hr = [], []
    for j, (t_send, t_recv) in enumerate(zip(last, spare)):
        tag = tag_kind * 1_000_000 + 1000 * j + step
        hs.append(comm.isend(t_send, place.next, tag))
        hr.append(comm.irecv(t_recv, place.prev, tag))
    return hs, hr


def _finish(comm, place: RingPlacement, handles, step: int):
    hs, hr = handles
    for h in hr:
        comm.wait(h, step, place.prev)
    for h in hs:
        comm.wait(h, step, place.next)


def _rotate(comm, place: RingPlacement, hold: list, spare, step: int, tag_kind: int):
    """Move every held chunk one ring rank on: hold[-1] goes to the next
    process, the previous process's last one lands in `spare`.  Returns the
    rotated list and the freed chunk (the new spare)."""
    _finish(comm, place, _post(comm, place, hold[-1], spare, step, tag_kind), step)
    return [spare] + hold[:-1], hold[-1]


def ring_forward(comm, kernels, place: RingPlacement, q, kv, o_out, lse_out):
    """Ring attention forward of this process's ring ranks.

    q[i]: [U][T][Hq/U][d] queries of local ring rank i (head-sharded when U > 1);
    kv[i]: (K, V), each [U][T][Hkv/U][d], its chunk, which travels;
    o_out[i] [U][T][Hq/U][d], lse_out[i] [U][Hq/U][T]: merged results.
    Per step s, local attention rank (r0+i)*U + u computes its partial with
    the chunk it holds (that of ring rank (r0+i-s) mod R) while the next
    chunk is in flight; the R partials are merged in step order at the end.
    `kv` buffers are rotated in place of one another: on return their
    contents are the chunks of other ranks."""
    R, U, Rl = place.R, place.U, place.Rl
    hold = [tuple(c) for c in kv]
    spare = tuple(kernels.empty_like(t) for t in kv[0])
    parts = [[kernels.partial_buffers(q[i][u], R) for u in range(U)] for i in range(Rl)]
    for s in range(R):
        comm.check_abort(s)
        handles = _post(comm, place, hold[-1], spare, s, TAG_KV) if s < R - 1 else None
        for i in range(Rl):
            for u in range(U):
                a = (place.r0 + i) * U + u
                o_p, l_p = parts[i][u]
                kernels.fwd_step(a, s, q[i][u], hold[i][0][u], hold[i][1][u], o_p[s], l_p[s])
        if handles is not None:
            _finish(comm, place, handles, s)
            hold, spare = [spare] + hold[:-1], hold[-1]
    for i in range(Rl):
        for u in range(U):
            o_p, l_p = parts[i][u]
            kernels.merge(o_p, l_p, o_out[i][u], lse_out[i][u])


def ring_backward(comm, kernels, place: RingPlacement, q, kv, o, lse, do, dq_out):
    """Ring attention backward of this process's ring ranks (same layouts
    as ring_forward; o [U][T][Hq/U][d], lse [U][Hq/U][T], do like q).

    Per step s each local attention rank computes its dQ contribution from
    the chunk it holds and the chunk's dK, dV contributions from its queries
    (step 0 writes them, later steps add to them); the chunk's K/V move on
    before the step (overlapping it), its fp32 dK/dV buffer after it.
    After the last step one more move brings every chunk's dK/dV back to its
    owner.  dq_out[i] [U][T][Hq/U][d] receives local ring rank i's dQ;
    returns, per local ring rank, its own chunk's (dK, dV), each
    [U][T][Hkv/U][d] fp32."""
    R, U, Rl = place.R, place.U, place.Rl
    stats = [[kernels.delta(o[i][u], do[i][u], lse[i][u]) for u in range(U)] for i in range(Rl)]
    hold = [tuple(c) for c in kv]
    spare = tuple(kernels.empty_like(t) for t in kv[0])
    ghold = [tuple(kernels.grad_buffer(t) for t in kv[0]) for _ in range(Rl)]
    gspare = tuple(kernels.grad_buffer(t) for t in kv[0])
    for s in range(R):
        comm.check_abort(s)
        handles = _post(comm, place, hold[-1], spare, s, TAG_KV) if s < R - 1 else None
        for i in range(Rl):
            for u in range(U):
                a = (place.r0 + i) * U + u
                kernels.bwd_step(a, s, q[i][u], do[i][u], stats[i][u], hold[i][0][u], hold[i][1][u],
                                 dq_out[i][u], ghold[i][0][u], ghold[i][1][u])
        if handles is not None:
            _finish(comm, place, handles, s)
            hold, spare = [spare] + hold[:-1], hold[-1]
        # The gradients of the chunks just computed follow them (after the
        # last step: home to their owners).
        ghold, gspare = _rotate(comm, place, ghold, gspare, s, TAG_GRAD)
    return ghold


class CudaRingKernels:
    """Per-step arithmetic on the GPU through the library's C ABI, on the
    current CUDA stream.  `plan` is the global plan (all R ring ranks)."""

    def __init__(self, plan, stream=None):
        import context_long_sequence_gb300 as cpa
        self.cpa = cpa
        self.plan = plan
        self.stream = stream

    @staticmethod
    def empty_like(t):
        return torch.empty_like(t)

    @staticmethod
    def grad_buffer(t):
        """fp32 gradient buffer of the shape of K or V, travelling with the chunk."""
        return torch.empty(t.shape, dtype=torch.float32, device=t.device)

    def partial_buffers(self, q_a, R):
        T, Hl, d = q_a.shape
        return (torch.empty(R, T, Hl, d, dtype=torch.float32, device=q_a.device),
                torch.empty(R, Hl, T, dtype=torch.float32, device=q_a.device))

    def fwd_step(self, a, s, q_a, k_c, v_c, o_part, lse_part):
        self.cpa.cp_attn_fwd_step(self.plan, a, s, q_a, k_c, v_c, o_part, lse_part, stream=self.stream)

    def merge(self, o_parts, lse_parts, o_out, lse_out):
        R, T, Hl, d = o_parts.shape
        self.cpa.cp_merge_lse(R, T, Hl, d, o_parts, lse_parts, o_out, lse_out, stream=self.stream)

    def delta(self, o_a, do_a, lse_a):
        """The rank's row statistics (-LSE*log2e, -D) for its backward steps."""
        n = self.plan.workspace_size(self.cpa.CP_OP_BWD_RANK_STATS) // 4
        out = torch.empty(n, dtype=torch.float32, device=do_a.device)
        self.cpa.cp_attn_bwd_delta(self.plan, o_a, do_a, lse_a, out, stream=self.stream)
        return out

    def bwd_step(self, a, s, q_a, do_a, stats_a, k_c, v_c, dq_a, dk_c, dv_c):
        self.cpa.cp_attn_bwd_step(self.plan, a, s, q_a, do_a, stats_a, k_c, v_c, dq_a, dk_c, dv_c,
                                  stream=self.stream)
