"""The ring transport (context_long_sequence_gb300.transport) between real
processes: 2 and 4 gloo ranks on the CPU run the forward and backward
schedules, with the oracle doing each step's arithmetic, and must reproduce
the plain-definition attention and gradients for every ring rank and head
group (ring and USP placements, zigzag with documents).  Failures are made
on the host: a chunk that one rank never sends, and a rank that dies before
a step; every rank must end with a TransportError within a few wait limits.
"""
import os
import socket
import sys
import time

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


class OracleKernels:
    """The transport's per-step arithmetic done by the oracle (fp64, CPU)."""

    def __init__(self, oracle, L, R, U, layout, offsets):
        self.orc, self.R, self.U, self.offsets = oracle, R, U, offsets
        self.T = L // R
        self.pos = oracle.ring_positions(L, R, layout, offsets)

    def rank_pos(self, r):
        return self.pos[r * self.T:(r + 1) * self.T]

    @staticmethod
    def empty_like(t):
        return torch.empty_like(t)

    @staticmethod
    def grad_buffer(t):
        return torch.empty(t.shape, dtype=torch.float64)

    def partial_buffers(self, q_a, R):
        T, Hl, d = q_a.shape
        return torch.empty(R, T, Hl, d, dtype=torch.float64), torch.empty(R, Hl, T, dtype=torch.float64)

    def fwd_step(self, a, s, q_a, k_c, v_c, o_part, lse_part):
        r = a // self.U
        src = (r - s) % self.R
        O, LSE = self.orc.attention_rows(q_a.numpy(), k_c.numpy(), v_c.numpy(), q_pos=self.rank_pos(r),
                                         k_pos=self.rank_pos(src), offsets=self.offsets)
        o_part.copy_(torch.from_numpy(O))
        lse_part.copy_(torch.from_numpy(LSE))

    def merge(self, o_parts, lse_parts, o_out, lse_out):
        o, lse = self.orc.merge([(o_parts[s].numpy(), lse_parts[s].numpy()) for s in range(o_parts.shape[0])])
        o_out.copy_(torch.from_numpy(o))
        lse_out.copy_(torch.from_numpy(lse))

    def delta(self, o_a, do_a, lse_a):
        return o_a, lse_a  # the oracle's step forms D = rowsum(dO * O) from O itself

    def bwd_step(self, a, s, q_a, do_a, stats, k_c, v_c, dq_a, dk_c, dv_c):
        o_a, lse_a = stats
        r = a // self.U
        src = (r - s) % self.R
        pq, pk, pv = self.orc.attention_bwd_partial(q_a.numpy(), do_a.numpy(), o_a.numpy(), lse_a.numpy(),
                                                    k_c.numpy(), v_c.numpy(), self.rank_pos(r),
                                                    self.rank_pos(src), offsets=self.offsets)
        for out, val in ((dq_a, pq), (dk_c, pk), (dv_c, pv)):
            if s == 0:
                out.copy_(torch.from_numpy(val))
            else:
                out.add_(torch.from_numpy(val))


def _problem(case):
    L, Hq, Hkv, d, U, R, layout, offsets, seed = case
    rng = np.random.default_rng(seed)
    f = lambda *sh: torch.from_numpy(rng.standard_normal(sh)).to(torch.bfloat16).double().numpy()  # noqa: E731
    return f(L, Hq, d), f(L, Hkv, d), f(L, Hkv, d), f(L, Hq, d)


def _head_sharded(orc, x_slots, r, T, U):
    """[U][T][H/U][d] of ring rank r: its Ulysses group's seq->head exchange."""
    n = T // U
    return orc.ulysses_seq_to_head(x_slots[r * T:(r + 1) * T].reshape((U, n) + x_slots.shape[1:]), U)


def _lse_head_sharded(lse_full_slots, r, T, U):
    """[U][H/U][T] of ring rank r from LSE [H][slots]."""
    H = lse_full_slots.shape[0]
    return lse_full_slots[:, r * T:(r + 1) * T].reshape(U, H // U, T)


def _report(q_out, item):
    """Put a result and flush the queue before the process exits."""
    q_out.put(item)
    q_out.close()
    q_out.join_thread()


def _worker(rank, world, port, case, mode, q_out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import datetime

    import torch.distributed as dist

    import oracle
    from context_long_sequence_gb300 import transport as tr
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=30))
    try:
        L, Hq, Hkv, d, U, R, layout, offsets, seed = case
        q, k, v, do = _problem(case)
        kern = OracleKernels(oracle, L, R, U, layout, offsets)
        place = tr.RingPlacement(R=R, U=U, world=world, rank=rank)
        T = L // R
        pos = kern.pos
        qs, ks, vs, dos = (oracle.shard(x, pos) for x in (q, k, v, do))
        comm = tr.DistComm(timeout_s=2.0 if mode.startswith("fault") else 30.0)
        if mode == "fault_drop":
            real_isend = comm.isend

            def isend(t, peer, tag):   # rank 1 never sends its chunk of step 1
                if rank == 1 and tag % 1000 == 1 and tag // 1_000_000 == tr.TAG_KV:
                    return None
                return real_isend(t, peer, tag)
            comm.isend = isend
            real_wait = comm.wait
            comm.wait = lambda h, s, p: None if h is None else real_wait(h, s, p)
        rr = range(place.r0, place.r0 + place.Rl)
        Q = [torch.from_numpy(_head_sharded(oracle, qs, r, T, U)) for r in rr]
        KV = [(torch.from_numpy(_head_sharded(oracle, ks, r, T, U)), torch.from_numpy(_head_sharded(oracle, vs, r, T, U)))
              for r in rr]
        O_full, LSE_full = oracle.attention(q, k, v, offsets=offsets)
        Os, LSEs = oracle.shard(O_full, pos), LSE_full[:, pos]
        if mode == "fault_die" and rank == world - 1:
            os._exit(3)                # dies before its first step
        if mode in ("fwd", "fault_drop", "fault_die"):
            o_out = [torch.empty_like(x) for x in Q]
            lse_out = [torch.empty(U, Hq // U, T, dtype=torch.float64) for _ in rr]
            t0 = time.time()
            try:
                tr.ring_forward(comm, kern, place, Q, KV, o_out, lse_out)
            except tr.TransportError as e:
                _report(q_out, (rank, "error", e.kind, e.step, time.time() - t0))
                os._exit(0)
            if mode != "fwd":
                # Every chunk this rank needed arrived, so its own result is
                # complete; the failure elsewhere reaches it through the
                # store's abort flag, which it checks before its next call.
                while time.time() - t0 < 15.0:
                    try:
                        comm.check_abort(R)
                    except tr.TransportError as e:
                        _report(q_out, (rank, "error_before_next_call", e.kind, e.step, time.time() - t0))
                        os._exit(0)
                    time.sleep(0.05)
                _report(q_out, (rank, "finished", None, None, time.time() - t0))
                os._exit(0)
            err_o = max(float(np.abs(o_out[i].numpy() - _head_sharded(oracle, Os, r, T, U)).max())
                        for i, r in enumerate(rr))
            err_l = max(float(np.abs(lse_out[i].numpy() - _lse_head_sharded(LSEs, r, T, U)).max())
                        for i, r in enumerate(rr))
            _report(q_out, (rank, "ok", err_o, err_l, 0.0))
        else:
            _, _, dq_f, dk_f, dv_f = oracle.attention_bwd(q, k, v, do, offsets=offsets)
            dqs, dks, dvs = (oracle.shard(x, pos) for x in (dq_f, dk_f, dv_f))
            Oh = [torch.from_numpy(_head_sharded(oracle, Os, r, T, U)) for r in rr]
            Lh = [torch.from_numpy(np.ascontiguousarray(_lse_head_sharded(LSEs, r, T, U))) for r in rr]
            dOh = [torch.from_numpy(_head_sharded(oracle, dos, r, T, U)) for r in rr]
            dq_out = [torch.empty_like(x) for x in Q]
            dkv = tr.ring_backward(comm, kern, place, Q, KV, Oh, Lh, dOh, dq_out)
            err = 0.0
            for i, r in enumerate(rr):
                err = max(err, float(np.abs(dq_out[i].numpy() - _head_sharded(oracle, dqs, r, T, U)).max()))
                err = max(err, float(np.abs(dkv[i][0].numpy() - _head_sharded(oracle, dks, r, T, U)).max()))
                err = max(err, float(np.abs(dkv[i][1].numpy() - _head_sharded(oracle, dvs, r, T, U)).max()))
            _report(q_out, (rank, "ok", err, 0.0, 0.0))
    except Exception as e:  # reported to the parent
        _report(q_out, (rank, "exception", repr(e)[:300], None, 0.0))
    os._exit(0)


def _run(world, case, mode, timeout=120):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, case, mode, q)) for r in range(world)]
    for p in procs:
        p.start()
    expect = world - (1 if mode == "fault_die" else 0)
    out = {}
    deadline = time.time() + timeout
    while len(out) < expect and time.time() < deadline:
        try:
            r, *rest = q.get(timeout=max(1.0, deadline - time.time()))
            out[r] = rest
        except Exception:
            break
    for p in procs:
        p.join(timeout=30)
        if p.is_alive():
            p.kill()
    return out


# L, Hq, Hkv, d, U, R, layout, offsets, seed
CASES = {
    "ring_R4_zigzag_docs": (96, 4, 2, 8, 1, 4, 1, [0, 30, 31, 96], 1),
    "usp_U2xR4_contig": (128, 4, 2, 8, 2, 4, 0, None, 2),
}


@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("name", sorted(CASES))
def test_ring_forward_over_gloo_matches_oracle(world, name):
    out = _run(world, CASES[name], "fwd")
    assert sorted(out) == list(range(world)), out
    for r, (status, eo, el, _) in out.items():
        assert status == "ok", (r, status, eo)
        assert eo < 1e-12 and el < 1e-12, (r, eo, el)


@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("name", sorted(CASES))
def test_ring_backward_over_gloo_matches_oracle(world, name):
    out = _run(world, CASES[name], "bwd")
    assert sorted(out) == list(range(world)), out
    for r, (status, err, _, _) in out.items():
        assert status == "ok", (r, status, err)
        assert err < 1e-11, (r, err)


def test_dropped_chunk_aborts_every_rank():
    """Rank 1 never sends its step-1 chunk: rank 2 times out waiting for it
    (2 s limit) and raises the abort.  Every other rank either fails a
    later wait or, if all its own chunks arrived, sees the abort flag before
    its next call; none goes on unaware."""
    out = _run(4, CASES["ring_R4_zigzag_docs"], "fault_drop")
    assert sorted(out) == [0, 1, 2, 3], out
    kinds = {r: v[1] for r, v in out.items()}
    assert all(v[0] in ("error", "error_before_next_call") for v in out.values()), out
    assert out[2][0] == "error" and kinds[2] == "timeout" and out[2][2] == 1, out
    assert all(v[3] < 20.0 for v in out.values()), out


def test_dead_rank_aborts_the_others():
    """The last rank exits before its first step: the others end with a
    TransportError within a few wait limits instead of hanging."""
    out = _run(4, CASES["ring_R4_zigzag_docs"], "fault_die")
    assert sorted(out) == [0, 1, 2], out
    assert all(v[0] in ("error", "error_before_next_call") for v in out.values()), out
    assert any(v[0] == "error" for v in out.values()), out
    assert all(v[3] < 20.0 for v in out.values()), out
