#!/usr/bin/env python
"""Benchmark of causal context-parallel attention forward on GB300.

One step = one cp_attn_fwd call over the whole workload (every emulated
rank): with Ulysses, the seq->head reshard of Q, K, V, the per-head-group
ring attention and the head->seq reshard of O and LSE; with emit-partials,
the per-step partials and their merge.  Inputs are seeded synthetic bf16
N(0,1) tensors resident in HBM; L2 is flushed (a 256 MiB write) before every
timed step and the flush is outside the step's CUDA-event bracket.

The default workload is the largest one that fits one GPU: USP (Ulysses 4 x
ring 8, zigzag) over L = 1,048,576 tokens.  Before it, the other four
workloads are measured in the same run (``per_config``): the 1K-token
emit-partials ring, the 16K Ulysses forward, the 64K zigzag ring forward
with its backward, and the 128K packed-document ring.

Prints one JSON line.  ``value`` is useful TFLOP/s (4 * d * Hq * visible
(query, key) pairs per step, summed over ranks, / the max-over-ranks time).
``--impl reference`` times the CPU oracle instead, on bounded samples of the
same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

DEFAULT_WORKLOAD = "usp_fwd_L1M_U4xR8_zigzag"
METRIC = "CP causal attn fwd TFLOPS & tokens/s, L=1K-1M, % of GB300 bf16 dense peak"
BWD_FLOP_RATIO = 2.5   # backward useful FLOPs per forward FLOP (dV, dP, dQ, dK products + recompute of S excluded)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SUSTAINED_MS = 1000.0  # launches this long run under the power cap: compared with the sustained tensor peak
TIMED_WORK_S = 5.0     # target seconds of GPU work for secondary repeated measurements


def useful_flops(w: workloads.Workload, offsets) -> int:
    """4 * d * Hq * (visible pairs): QK^T and PV, 2 FLOPs per multiply-add."""
    if offsets is None:
        pairs = w.L * (w.L + 1) // 2
    else:
        lens = np.diff(np.asarray(offsets, dtype=np.int64))
        pairs = int((lens * (lens + 1) // 2).sum())
    return 4 * w.d * w.Hq * pairs


def row_visible(pos: np.ndarray, offsets) -> np.ndarray:
    if offsets is None:
        return pos + 1
    offs = np.asarray(offsets, dtype=np.int64)
    start = offs[np.searchsorted(offs, pos, side="right") - 1]
    return pos - start + 1


LAYOUT_NAMES = ["contiguous", "zigzag", "balanced"]


def workload_config(w, offsets, args, world: int, positions) -> dict:
    """The `config` object of the JSON line (both arms print the same one).
    positions: the slot -> global position map of the plan."""
    layout = LAYOUT_NAMES[w.layout] + (f" (m={args.chunks_per_rank})" if w.layout == 2 else "")
    return {"workload": w.name, "L": w.L, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "ulysses": w.ulysses, "ring": w.ring,
            "layout": layout,
            "rank_work_spread": rank_work_spread(positions, w.ring, offsets),
            "kv_exchange": args.kv_exchange,
            "docs": bool(offsets is not None),
            "num_docs": 0 if offsets is None else len(offsets) - 1, "P": w.P,
            "parallelism": f"replicas x{world} (all {w.P} CP ranks emulated per GPU)",
            "step": "forward + backward" if w.backward else "forward",
            "l2": "flushed (256 MiB write) before every timed step"}


def rank_work_spread(index_map, R: int, offsets) -> float:
    """max / mean over ring ranks of the visible (query, key) pairs whose
    query the rank holds: a query at position i sees i - doc_start(i) + 1 keys."""
    pos = np.asarray(index_map, dtype=np.int64)
    row_keys = row_visible(pos, offsets)
    work = row_keys.reshape(R, -1).sum(axis=1).astype(np.float64)
    return round(float(work.max() / work.mean()), 4)


def secondary_bounds(ex2_per_clk, mma_clk, n_sm, clock_rec, d):
    """The exp2 (MUFU) bound and the tensor rate of a plain MMA stream, at the
    GPU's maximum SM clock: every visible (query, key) pair of a head costs one
    exp2 and 4*d useful FLOPs."""
    mhz = (clock_rec or {}).get("sm_max_mhz") or 2070.0
    hz = float(mhz) * 1e6
    return {"ex2_per_clk_per_sm": round(ex2_per_clk, 2), "mma_clk_m128n128k16": round(mma_clk, 2),
            "sm_count": n_sm, "sm_clock_mhz": mhz,
            "exp2_bound_tflops": round(ex2_per_clk * n_sm * hz * 4 * d / 1e12, 1),
            "mma_stream_tflops": round(n_sm * hz * 2 * 128 * 128 * 16 / mma_clk / 1e12, 1)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(path):
        return dict(FALLBACK_PEAKS), "fallback"
    try:
        raw = json.load(open(path))
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"
    flat = {}

    def walk(x):
        if isinstance(x, dict):
            for k, v in x.items():
                if isinstance(v, (int, float)) and not isinstance(v, bool):
                    flat.setdefault(k, float(v))
                else:
                    walk(v)
    walk(raw)
    out = {}
    for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
        out[key] = flat.get(key, FALLBACK_PEAKS[key])
    return out, "measured" if all(k in flat for k in ("hbm_gbs", "bf16_tflops")) else "partly fallback"


def tensor_peak(peaks, peak_src, launch_ms):
    """(peak TFLOP/s, its label) for an attention launch of launch_ms: the
    sustained peak for launches of a second or more, else the burst one."""
    sustained = launch_ms >= SUSTAINED_MS
    return (peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"],
            f"bf16 dense {'sustained' if sustained else 'burst'}, {peak_src}")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            try:
                power.append(float(f[3]))
            except ValueError:
                pass
            for n, flag in zip(names, f[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(n)
        rec = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
               "reasons": sorted(reasons), "samples": len(sm)}
        if power:
            rec["power_w_median"] = statistics.median(power)
        return rec


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("attn_fwd.cu", "ptx.cuh", "kernels.h", "debug.cuh", "tmap.h"):
        h.update(open(os.path.join(ROOT, "context_long_sequence_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per attention launch from a committed ncu capture, if the
    kernel source has not changed since (else None), with how it was taken."""
    path = os.path.join(ROOT, "profiles", "attn_fwd_traffic.json")
    if not os.path.exists(path):
        return None, None
    try:
        rec = json.load(open(path))
    except Exception:
        return None, None
    if rec.get("kernel_source_sha") != kernel_source_hash():
        return None, "kernel changed since the committed capture"
    entry = rec.get("per_launch_bytes", {}).get(workload)
    if entry is None:
        return None, None
    if isinstance(entry, dict):
        return entry.get("bytes"), entry.get("how")
    return entry, rec.get("source")


def sha256_tensors(tensors: dict) -> dict:
    """SHA-256 of each (CPU) tensor's bytes, hashed in parallel threads."""
    out = {}

    def one(name, t):
        h = hashlib.sha256()
        raw = t.contiguous().view(-1).view(dtype=__import__("torch").uint8).numpy()
        step = 1 << 28
        for i in range(0, raw.size, step):
            h.update(memoryview(raw[i:i + step]))
        out[name] = h.hexdigest()

    threads = [threading.Thread(target=one, args=(n, t)) for n, t in tensors.items()]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    return {n: out[n] for n in tensors}


def run_metadata(dev, w):
    import torch
    props = torch.cuda.get_device_properties(dev)
    meta = {"seed": w.seed, "gpu_name": props.name, "sm_count": props.multi_processor_count,
            "torch": torch.__version__, "cuda_runtime": torch.version.cuda,
            "host_cores": len(os.sched_getaffinity(0))}
    try:
        drv = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout.strip().splitlines()
        meta["driver"] = drv[0] if drv else None
    except Exception:
        meta["driver"] = None
    return meta


# ---------------------------------------------------------------------------- CPU oracle timing


def oracle_rows_per_call(L: int, cap: int) -> int:
    """Query rows per oracle call: about 2^22 scores per call (fewer rows at long L)."""
    return max(1, min(cap, (1 << 22) // L))


def time_oracle(w, inputs_cpu, offsets, rows_per_call, heads, seed, min_seconds, max_calls=64):
    """Time the oracle on seeded random query rows until at least min_seconds."""
    import oracle
    rng = np.random.default_rng(seed)
    flops = 0
    t0 = time.perf_counter()
    calls = 0
    while True:
        rows = np.sort(rng.choice(w.L, size=rows_per_call, replace=False))
        oracle.attention_rows(inputs_cpu["q"], inputs_cpu["k"], inputs_cpu["v"], rows=rows, offsets=offsets,
                              heads=heads)
        flops += 4 * w.d * len(heads) * int(row_visible(rows, offsets).sum())
        calls += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or calls >= max_calls:
            return flops, el, calls


def cpu_inputs(w):
    return workloads.make_inputs(w.L, w.Hq, w.Hkv, w.d, w.seed, device="cpu", k_scale=w.k_scale)


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise max of per-rank timings (the job is as slow as its
    slowest replica).  The only collective besides the barriers."""
    import torch
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def aggregate_value(flops_per_step_per_rank: int, world: int, ms_per_step_max: float) -> float:
    """Whole-job useful TFLOP/s: every rank's work over the slowest rank's time."""
    return world * flops_per_step_per_rank / (ms_per_step_max * 1e-3) / 1e12


def reps_for(step_ms: float, cap: int) -> int:
    """Repetitions of a secondary measurement: about TIMED_WORK_S of GPU
    work, at least 3 and at most cap."""
    return int(max(3, min(cap, math.ceil(TIMED_WORK_S * 1e3 / max(step_ms, 1e-3)))))


def make_plan(cpa, w, offsets, chunks_per_rank=8, kv_exchange="ring", out_fp32=False):
    return cpa.Plan(w.L, w.Hq, w.Hkv, w.d, ulysses_degree=w.ulysses, ring_degree=w.ring, layout=w.layout,
                    doc_offsets=offsets, emit_partials=w.emit_partials, chunks_per_rank=chunks_per_rank,
                    kv_exchange=cpa.CP_KV_ALLGATHER if kv_exchange == "allgather" else cpa.CP_KV_RING,
                    out_fp32=out_fp32)


class Timer:
    """CUDA-event timing on the launching stream, L2 flushed before each rep."""

    def __init__(self, torch, dev, stream, flush):
        self.torch, self.dev, self.stream, self.flush = torch, dev, stream, flush

    def __call__(self, fn, reps):
        torch = self.torch
        ts = []
        for _ in range(reps):
            self.flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(self.stream)
            fn()
            b.record(self.stream)
            torch.cuda.synchronize(self.dev)
            ts.append(a.elapsed_time(b))
        return statistics.mean(ts)


def measure_other_workload(cpa, torch, w, dev, timer, peaks, peak_src):
    """Forward (and, for the ring fwd+bwd workload, backward) of one more
    workload, on its own seeded inputs: 3 warm-up calls, then the mean of
    about TIMED_WORK_S of repetitions, L2 flushed before each."""
    offsets = workloads.workload_doc_offsets(w)
    plan = make_plan(cpa, w, offsets)
    g = workloads.make_inputs(w.L, w.Hq, w.Hkv, w.d, w.seed, device=dev, k_scale=w.k_scale, with_do=w.backward)
    idx = torch.from_numpy(plan.index_map().astype(np.int64)).to(dev)
    q, k, v = (g[n][idx].contiguous() for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(plan.P, w.Hq, plan.n, dtype=torch.float32, device=dev)
    ws = cpa.alloc_workspace(plan, device=dev)
    stream = timer.stream

    def fwd():
        cpa.cp_attn_fwd(plan, q, k, v, o, lse, ws, stream=stream)

    for _ in range(3):
        fwd()
    torch.cuda.synchronize(dev)
    t1 = timer(fwd, 1)
    fwd_ms = timer(fwd, reps_for(t1, 50))
    flops = useful_flops(w, offsets)
    peak, plabel = tensor_peak(peaks, peak_src, fwd_ms)
    rec = {"L": w.L, "P": w.P, "ulysses": w.ulysses, "ring": w.ring, "layout": LAYOUT_NAMES[w.layout],
           "docs": 0 if offsets is None else len(offsets) - 1, "useful_flops_fwd": flops,
           "fwd_ms": round(fwd_ms, 4), "fwd_tflops": round(flops / fwd_ms / 1e9, 2),
           "fwd_frac": round(flops / fwd_ms / 1e9 / peak, 4), "peak": peak, "peak_source": plabel,
           "tokens_per_s": round(w.L / (fwd_ms * 1e-3), 1),
           "step": "emit-partials + merge" if w.emit_partials else
                   ("attention; Ulysses exchanges in its loads and stores" if w.ulysses > 1
                    else "attention (fused merge)")}
    if w.backward:
        do = g["do"][idx].contiguous()
        dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
        dk = torch.empty(k.shape, dtype=torch.float32, device=dev)
        dv = torch.empty(v.shape, dtype=torch.float32, device=dev)
        ws_b = cpa.alloc_workspace(plan, cpa.CP_OP_BWD, device=dev)

        def bwd():
            cpa.cp_attn_bwd(plan, q, k, v, o, lse, do, dq, dk, dv, ws_b, stream=stream)

        for _ in range(2):
            bwd()
        torch.cuda.synchronize(dev)
        bwd_ms = timer(bwd, reps_for(timer(bwd, 1), 30))
        bflops = flops * BWD_FLOP_RATIO
        bpeak, bplabel = tensor_peak(peaks, peak_src, bwd_ms)
        rec.update({"bwd_ms": round(bwd_ms, 4), "bwd_tflops": round(bflops / bwd_ms / 1e9, 2),
                    "bwd_frac": round(bflops / bwd_ms / 1e9 / bpeak, 4), "bwd_peak_source": bplabel,
                    "fwd_bwd_ms": round(fwd_ms + bwd_ms, 4),
                    "fwd_bwd_tflops": round((flops + bflops) / (fwd_ms + bwd_ms) / 1e9, 2)})
        del do, dq, dk, dv, ws_b
    if cpa.cp_get_status(stream) != 0:
        raise RuntimeError(f"device status set while measuring {w.name}")
    del q, k, v, o, lse, ws, g
    torch.cuda.empty_cache()
    return rec


# ---------------------------------------------------------------------------- main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=[w.name for w in workloads.WORKLOADS])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-full", action="store_true",
                    help="the CPU baseline runs the oracle over every query row and head (minutes at L=16K) "
                         "instead of a sample")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the measurements of the other four workloads after the main one")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end measurement")
    ap.add_argument("--no-hash", action="store_true", help="skip the SHA-256 of the inputs")
    ap.add_argument("--layout", choices=["workload", "contiguous", "zigzag", "balanced"], default="workload",
                    help="token layout of the ring shards (default: the workload's own)")
    ap.add_argument("--chunks-per-rank", type=int, default=8, help="chunks per ring rank of the balanced layout")
    ap.add_argument("--kv-exchange", choices=["ring", "allgather"], default="ring",
                    help="how ranks obtain the other ranks' K/V (all-gather: ring plans with U == 1 only)")
    ap.add_argument("--backward", action="store_true",
                    help="add the backward to every step (the ring fwd+bwd workload always has it)")
    ap.add_argument("--transport", action="store_true",
                    help="with one GPU: run the multi-GPU ring-transport step (per-step launches, chunks "
                         "rotated through a loopback) instead of the single-launch step")
    ap.add_argument("--L", type=int, default=0,
                    help="override the workload's sequence length (small cases for profiling); 0 keeps it")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = workloads.WORKLOAD_BY_NAME[args.workload]
    if args.L:
        w = dataclasses.replace(w, L=args.L)
    if args.backward:
        w = dataclasses.replace(w, backward=True)
    if args.layout != "workload":
        w = dataclasses.replace(w, layout={"contiguous": 0, "zigzag": 1, "balanced": 2}[args.layout])
    offsets = workloads.workload_doc_offsets(w)
    flops_fwd = useful_flops(w, offsets)
    flops_step = int(flops_fwd * (1 + BWD_FLOP_RATIO)) if w.backward else flops_fwd
    warmup = max(3, args.warmup)

    if args.impl == "reference":
        if rank != 0:
            return 0
        return run_reference(args, w, offsets, flops_step, warmup, world)

    import torch
    import context_long_sequence_gb300 as cpa
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank)
    if (world > 1 or args.transport) and transport_eligible(w, args, world):
        return run_transport(args, w, offsets, flops_fwd, flops_step, warmup, world, rank, dev, dist)

    # The other workloads first, each on its own buffers, freed before the
    # default workload's inputs are drawn.  Each is timed over up to 50
    # back-to-back launches (about half a second of work), long enough for
    # the power cap to act on the larger ones.
    per_config = {}
    if not args.no_per_config and not args.L and rank == 0:
        flush0 = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        timer0 = Timer(torch, dev, torch.cuda.current_stream(dev), flush0)
        peaks0, peak_src0 = load_peaks()
        for ow in workloads.WORKLOADS:
            if ow.name == w.name:
                continue
            per_config[ow.name] = measure_other_workload(cpa, torch, ow, dev, timer0, peaks0, peak_src0)
        del flush0, timer0
        torch.cuda.empty_cache()

    plan = make_plan(cpa, w, offsets, args.chunks_per_rank, args.kv_exchange)
    # Independent replica per GPU (the emulated ranks all live on one GPU):
    # each rank draws its own sequence.
    g_inputs = workloads.make_inputs(w.L, w.Hq, w.Hkv, w.d, w.seed + 7919 * rank, device=dev, k_scale=w.k_scale,
                                     with_do=w.backward)
    idx = torch.from_numpy(plan.index_map().astype(np.int64)).to(dev)
    q, k, v = (g_inputs[n][idx].contiguous() for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(plan.P, w.Hq, plan.n, dtype=torch.float32, device=dev)
    ws = cpa.alloc_workspace(plan, device=dev)
    if w.backward:
        do = g_inputs["do"][idx].contiguous()
        dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
        dk = torch.empty(k.shape, dtype=torch.float32, device=dev)
        dv = torch.empty(v.shape, dtype=torch.float32, device=dev)
        ws_bwd = cpa.alloc_workspace(plan, cpa.CP_OP_BWD, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    timer = Timer(torch, dev, stream, flush)
    # The rates behind the secondary bounds: exp2 per SM clock (one per
    # visible pair and head) and clocks per M128 N128 K16 MMA, measured here.
    ex2_per_clk, mma_clk = cpa.cp_measure_rates(stream=stream)
    # And the fixed cost of a barrier check in the MMA-issuing warps.
    bar_clk = cpa.cp_measure_barrier_check(stream=stream)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count

    def fwd():
        cpa.cp_attn_fwd(plan, q, k, v, o, lse, ws, stream=stream)

    def bwd():
        cpa.cp_attn_bwd(plan, q, k, v, o, lse, do, dq, dk, dv, ws_bwd, stream=stream)

    def step():
        fwd()
        if w.backward:
            bwd()

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    status = cpa.cp_get_status(stream)
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    clocks = ClockSampler(local_rank)
    # Per timed step: events around the whole step and, inside it, around
    # the forward (when the forward is the attention launch alone, its
    # duration is the kernel's, measured live over the timed region).
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(args.steps)]
    barrier()
    clocks.start()
    t_wall = time.perf_counter()
    for e0, ef, e1 in evs:
        flush.zero_()
        e0.record(stream)
        fwd()
        ef.record(stream)
        if w.backward:
            bwd()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall
    clock_rec = clocks.stop()
    barrier()
    step_ms = [e0.elapsed_time(e1) for e0, _, e1 in evs]
    fwd_live_ms = statistics.mean(e0.elapsed_time(ef) for e0, ef, _ in evs) if evs else float("nan")
    total_ms = sum(step_ms)
    mean_step_ms = total_ms / max(1, args.steps)
    if cpa.cp_get_status(stream) != 0:
        raise RuntimeError("device status set during the timed region")

    # ---- end to end through the public API with host buffers
    # Every step copies its inputs from pinned host memory and its results
    # back.  Pipelined: two device buffer sets, host->device copies on one
    # stream and device->host copies on another, so the copies of
    # neighbouring steps overlap the computation of this one (the way a
    # training loop feeds the GPU).  The serial figure (copy in, compute,
    # copy out, one step after the other on one stream) is reported too.
    in_names = ["q", "k", "v"] + (["do"] if w.backward else [])
    out_names = ["o", "lse"] + (["dq", "dk", "dv"] if w.backward else [])
    set0 = {"q": q, "k": k, "v": v, "o": o, "lse": lse}
    if w.backward:
        set0.update(do=do, dq=dq, dk=dk, dv=dv)
    e2e_steps = reps_for(mean_step_ms, 10)
    # The pipeline's first copy in and last copy out are not overlapped:
    # at least six steps, so that they weigh as in a run of many.
    e2e_pipe_steps = max(6, e2e_steps)
    e2e_ms = e2e_serial_ms = float("nan")
    h2d = sum(set0[n].numel() * set0[n].element_size() for n in in_names)
    d2h = sum(set0[n].numel() * set0[n].element_size() for n in out_names)
    if not args.no_e2e:
        sets = [set0, {n: torch.empty_like(t) for n, t in set0.items()}]
        host_in = {n: set0[n].cpu().pin_memory() for n in in_names}
        host_out = [{n: torch.empty(set0[n].shape, dtype=set0[n].dtype).pin_memory() for n in out_names}
                    for _ in range(2)]

        def step_on(b):
            S = sets[b]
            cpa.cp_attn_fwd(plan, S["q"], S["k"], S["v"], S["o"], S["lse"], ws, stream=stream)
            if w.backward:
                cpa.cp_attn_bwd(plan, S["q"], S["k"], S["v"], S["o"], S["lse"], S["do"], S["dq"], S["dk"], S["dv"],
                                ws_bwd, stream=stream)

        s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in, ev_comp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

        def pipelined(nsteps):
            s_h2d.wait_stream(stream)
            e0 = torch.cuda.Event(enable_timing=True)
            e0.record(s_h2d)
            for i in range(nsteps):
                b = i % 2
                if i >= 2:
                    s_h2d.wait_event(ev_comp[b])     # step i-2 no longer reads these inputs
                with torch.cuda.stream(s_h2d):
                    for n in in_names:
                        sets[b][n].copy_(host_in[n], non_blocking=True)
                ev_in[b].record(s_h2d)
                stream.wait_event(ev_in[b])
                if i >= 2:
                    stream.wait_event(ev_out[b])     # step i-2's results have left these buffers
                step_on(b)
                ev_comp[b].record(stream)
                s_d2h.wait_event(ev_comp[b])
                with torch.cuda.stream(s_d2h):
                    for n in out_names:
                        host_out[b][n].copy_(sets[b][n], non_blocking=True)
                ev_out[b].record(s_d2h)
            e1 = torch.cuda.Event(enable_timing=True)
            e1.record(s_d2h)                         # after the last copy, which follows everything
            torch.cuda.synchronize(dev)
            return e0.elapsed_time(e1)

        def serial_step():
            for n in in_names:
                set0[n].copy_(host_in[n], non_blocking=True)
            step_on(0)
            for n in out_names:
                host_out[0][n].copy_(set0[n], non_blocking=True)

        pipelined(2)
        barrier()
        e2e_ms = pipelined(e2e_pipe_steps) / e2e_pipe_steps
        serial_step()
        barrier()
        ee0, ee1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ee0.record(stream)
        for _ in range(e2e_steps):
            serial_step()
        ee1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_serial_ms = ee0.elapsed_time(ee1) / e2e_steps
        del sets, host_in, host_out

    # ---- per-kernel breakdown (the dominant kernel's roofline)
    kern = {}
    U, R = w.ulysses, w.ring
    if U > 1:
        qh = torch.empty(R, U, plan.L // R, w.Hq // U, w.d, dtype=torch.bfloat16, device=dev)
        kh = torch.empty(R, U, plan.L // R, w.Hkv // U, w.d, dtype=torch.bfloat16, device=dev)
        vh = torch.empty_like(kh)
        oh = torch.empty_like(qh)
        lh = torch.empty(R, U, w.Hq // U, plan.L // R, dtype=torch.float32, device=dev)
    else:
        qh, kh, vh, oh, lh = q, k, v, o, lse
        if args.kv_exchange == "allgather":  # the attention alone reads the gathered K/V (position order)
            kh, vh = g_inputs["k"], g_inputs["v"]

    reps = reps_for(mean_step_ms, 10)
    if U > 1:
        # The forward is one launch (the Ulysses exchanges are the kernel's
        # addressing): the attention alone is cp_attn_fwd itself.
        attn_ms = timer(fwd, reps)
    else:
        attn_ms = timer(lambda: cpa.cp_attn_fwd_local(plan, qh, kh, vh, oh, lh, stream=stream), reps)
    kern["attn_fwd"] = {"ms": attn_ms, "tflops": flops_fwd / attn_ms / 1e9, "reps": reps}
    if U == 1 and not w.emit_partials:
        # Each ring rank's share alone (cp_attn_fwd_rank): the forward time of
        # one GPU per rank, communication aside, is the slowest rank's.
        per_rank = [timer(lambda r=r: cpa.cp_attn_fwd_rank(plan, r, q, kh, vh, o, lse, stream=stream), reps)
                    for r in range(R)]
        kern["attn_fwd_per_rank"] = {"ms": [round(t, 4) for t in per_rank], "max_ms": max(per_rank),
                                     "max_over_mean": max(per_rank) / statistics.mean(per_rank)}
    if w.backward:
        bwd_ms = timer(bwd, reps)
        kern["attn_bwd"] = {"ms": bwd_ms, "tflops": flops_fwd * BWD_FLOP_RATIO / bwd_ms / 1e9,
                            "kernels": "bwd_delta, attn_bwd_dkv, attn_bwd_dq"}
    if U > 1:
        # The two exchanges as copies (ulysses_reshard, the form the backward
        # and cp_attn_fwd_local callers use; the forward step folds them into
        # the attention's addressing): one launch for Q, K, V, one for O, LSE.
        def rin():
            cpa.ulysses_reshard_batch(plan, [(cpa.CP_SEQ_TO_HEAD, cpa.CP_TOKEN_MAJOR, w.Hq, w.d, 2, q, qh),
                                             (cpa.CP_SEQ_TO_HEAD, cpa.CP_TOKEN_MAJOR, w.Hkv, w.d, 2, k, kh),
                                             (cpa.CP_SEQ_TO_HEAD, cpa.CP_TOKEN_MAJOR, w.Hkv, w.d, 2, v, vh)],
                                      stream=stream)

        def rout():
            cpa.ulysses_reshard_batch(plan, [(cpa.CP_HEAD_TO_SEQ, cpa.CP_TOKEN_MAJOR, w.Hq, w.d, 2, oh, o),
                                             (cpa.CP_HEAD_TO_SEQ, cpa.CP_HEAD_MAJOR, w.Hq, 1, 4, lh, lse)],
                                      stream=stream)
        bytes_in = 2 * 2 * w.L * w.d * (w.Hq + 2 * w.Hkv)
        bytes_out = 2 * (2 * w.L * w.d * w.Hq + 4 * w.L * w.Hq)
        t_in = timer(rin, 10)
        t_out = timer(rout, 10)
        kern["reshard_seq_to_head"] = {"ms": t_in, "gbs": bytes_in / t_in / 1e6, "bytes": bytes_in}
        kern["reshard_head_to_seq"] = {"ms": t_out, "gbs": bytes_out / t_out / 1e6, "bytes": bytes_out}
    del qh, kh, vh, oh, lh

    # Standalone LSE merge at one ring rank's shape of the 64K ring workload
    # (8 ring-step partials of 8192 rows x 32 heads x 128): HBM-bound.
    mp, mr, mh, md = 8, 8192, 32, 128
    o_parts = torch.randn(mp, mr, mh, md, dtype=torch.float32, device=dev)
    lse_parts = torch.randn(mp, mh, mr, dtype=torch.float32, device=dev)
    o_m = torch.empty(mr, mh, md, dtype=torch.bfloat16, device=dev)
    lse_m = torch.empty(mh, mr, dtype=torch.float32, device=dev)
    t_merge = timer(lambda: cpa.cp_merge_lse(mp, mr, mh, md, o_parts, lse_parts, o_m, lse_m, stream=stream), 10)
    merge_bytes = mp * mr * mh * (4 * md + 4) + mr * mh * (2 * md + 4)
    kern["merge_8x8192x32x128"] = {"ms": t_merge, "gbs": merge_bytes / t_merge / 1e6, "bytes": merge_bytes}
    del o_parts, lse_parts, o_m, lse_m

    peaks, peak_src = load_peaks()
    total_ms, e2e_ms_max, e2e_serial_ms_max, attn_ms_max, fwd_live_ms = max_over_ranks(
        [total_ms, e2e_ms, e2e_serial_ms, attn_ms, fwd_live_ms], dist, dev)

    # Host copies of the global-order inputs: their SHA-256 and the oracle's
    # sample (rank 0 only).
    meta = None
    cpu = None
    if rank == 0:
        meta = run_metadata(dev, w)
        meta["seed"] = w.seed + 7919 * rank
        want_baseline = world == 1 and not args.no_cpu_baseline
        if want_baseline or not args.no_hash:
            cpu = {n: t.cpu() for n, t in g_inputs.items()}
        if not args.no_hash:
            meta["input_sha256"] = sha256_tensors(cpu)
            meta["input_sha256_of"] = "global-order bf16 tensors as drawn (before sharding), raw bytes"

    del q, k, v, o, lse, ws, g_inputs, set0
    if w.backward:
        del do, dq, dk, dv, ws_bwd
    torch.cuda.empty_cache()

    result = None
    if rank == 0:
        ms_per_step = total_ms / args.steps
        value = aggregate_value(flops_step, world, ms_per_step)
        # forward: attention (with U > 1 the Ulysses exchanges are its
        # addressing); merge with partials; two gathers with the all-gather
        # exchange.  backward: delta, dkv, dq (the exchanges again in their
        # addressing).
        launches_per_step = (1 + (1 if w.emit_partials else 0)
                             + (2 if args.kv_exchange == "allgather" else 0)
                             + (3 if w.backward else 0))
        # The attention kernel's duration: measured live over the timed
        # region when the forward is that one launch (fused merge, Ulysses
        # exchanges in its addressing); otherwise (a merge launch or the
        # all-gather copies beside it) the attention alone, timed after.
        fwd_launches = 1 + (1 if w.emit_partials else 0) + (2 if args.kv_exchange == "allgather" else 0)
        kern_ms = fwd_live_ms if fwd_launches == 1 else attn_ms
        kern_timing = ("CUDA events around the attention launch in every timed step" if fwd_launches == 1 else
                       "the attention alone, %d reps after the timed region" % kern.get("attn_fwd", {}).get("reps", 0))
        achieved = flops_fwd / (kern_ms * 1e-3) / 1e12
        peak, plabel = tensor_peak(peaks, peak_src, kern_ms)
        traffic, traffic_how = (None, None) if args.L else profiled_traffic(w.name)
        roofline = {"bound": "tensor", "kernel": "attn_fwd_kernel<%d>" % w.d, "achieved": round(achieved, 2),
                    "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "peak_source": plabel,
                    "traffic": traffic, "kernel_ms": round(kern_ms, 4), "timing": kern_timing}
        if traffic_how:
            roofline["traffic_source"] = traffic_how
        result = {
            "metric": METRIC,
            "value": round(value, 3),
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": warmup,
            "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": workload_config(w, offsets, args, world, plan.index_map()),
            "tokens_per_s": round(world * w.L / (ms_per_step * 1e-3), 1),
            "useful_flops_per_step": flops_step,
            "gpu_launches": launches_per_step * args.steps,
            "roofline": roofline,
            "kernels": {k_: {kk: (round(vv, 4) if isinstance(vv, float) else vv) for kk, vv in v_.items()}
                        for k_, v_ in kern.items()},
            "hbm_peak_gbs": peaks["hbm_gbs"],
            "secondary": dict(secondary_bounds(ex2_per_clk, mma_clk, n_sm, clock_rec, w.d),
                              barrier_check_clk=round(bar_clk, 1)),
            "clocks": clock_rec,
            "wall_s_timed": round(t_wall, 3),
        }
        if not args.no_e2e:
            result["e2e"] = {
                "value": round(world * flops_step / (e2e_ms_max * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms_max, 4),
                "steps": e2e_pipe_steps, "serial_steps": e2e_steps,
                "overlap": "2 device buffer sets; H2D and D2H of neighbouring steps overlap compute",
                "serial_value": round(world * flops_step / (e2e_serial_ms_max * 1e-3) / 1e12, 3),
                "serial_ms_per_step": round(e2e_serial_ms_max, 4)}
        if per_config:
            result["per_config"] = per_config
        if meta is not None:
            result["run"] = meta
        if world == 1 and not args.no_cpu_baseline and cpu is not None:
            result["cpu_baseline"] = cpu_baseline(w, cpu, offsets, flops_fwd, full=args.cpu_full)
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def transport_eligible(w, args, world) -> bool:
    """One sequence over `world` GPUs through the ring transport: ring plans
    (no emit-partials, no all-gather) whose ring degree the GPU count divides.
    Other cases run independent replicas."""
    return (not w.emit_partials and args.kv_exchange == "ring" and w.ring % world == 0 and not args.L)


def run_transport(args, w, offsets, flops_fwd, flops_step, warmup, world, rank, dev, dist):
    """N GPUs share one sequence (strong scaling): process p holds ring ranks
    [p*R/N, (p+1)*R/N) with all their Ulysses members; the Ulysses exchange is
    the library's reshard on the process's own slice, and the ring passes
    K/V chunks (and in the backward dK/dV) between processes through
    context_long_sequence_gb300.transport (NCCL point-to-point)."""
    import torch
    import context_long_sequence_gb300 as cpa
    from context_long_sequence_gb300 import transport as tr
    R, U, Rl = w.ring, w.ulysses, w.ring // world
    T, d = w.L // R, w.d
    plan = make_plan(cpa, w, offsets)
    # The reshard geometry of this process's slice: Rl ring groups of U members.
    local = cpa.Plan(Rl * T, w.Hq, w.Hkv, d, ulysses_degree=U, ring_degree=Rl)
    g = workloads.make_inputs(w.L, w.Hq, w.Hkv, d, w.seed, device=dev, k_scale=w.k_scale, with_do=w.backward)
    idx = torch.from_numpy(plan.index_map().astype(np.int64)).to(dev)
    sl = idx[rank * Rl * T:(rank + 1) * Rl * T]          # this process's slots (ring-rank major)
    q, k, v = (g[n][sl].contiguous() for n in ("q", "k", "v"))
    do = g["do"][sl].contiguous() if w.backward else None
    del g
    stream = torch.cuda.current_stream(dev)
    Hl, Hkl = w.Hq // U, w.Hkv // U
    qh = torch.empty(Rl, U, T, Hl, d, dtype=torch.bfloat16, device=dev)
    kh = torch.empty(Rl, U, T, Hkl, d, dtype=torch.bfloat16, device=dev)
    vh = torch.empty_like(kh)
    oh = torch.empty_like(qh)
    lh = torch.empty(Rl, U, Hl, T, dtype=torch.float32, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(Rl * U, w.Hq, T // U, dtype=torch.float32, device=dev)
    comm = tr.DistComm(timeout_s=600.0) if world > 1 else tr.LocalComm()
    kern = tr.CudaRingKernels(plan, stream=stream)
    place = tr.RingPlacement(R=R, U=U, world=world, rank=rank)
    if w.backward:
        doh = torch.empty_like(qh)
        dqh = torch.empty(Rl, U, T, Hl, d, dtype=torch.float32, device=dev)
        dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
        dk = torch.empty(k.shape, dtype=torch.float32, device=dev)
        dv = torch.empty(v.shape, dtype=torch.float32, device=dev)

    def reshard(jobs):
        if U > 1:
            cpa.ulysses_reshard_batch(local, jobs, stream=stream)

    def views(x):                                         # [Rl][U][T][..] per local ring rank
        return [x[i] for i in range(Rl)]

    if U == 1:                                            # head-sharded == sequence-sharded
        qh, oh = (x.view(Rl, 1, T, x.shape[1], d) for x in (q, o))
        lh = lse.view(Rl, 1, w.Hq, T)
        if w.backward:
            doh = do.view(Rl, 1, T, w.Hq, d)
            dqh = dq.view(Rl, 1, T, w.Hq, d)

    def stage_kv(extra=()):
        """K/V (and `extra` jobs) into the head-sharded chunk buffers, which
        the ring rotates (with U == 1 K/V travel in copies, not in the
        caller's own buffers)."""
        if U > 1:
            reshard([(cpa.CP_SEQ_TO_HEAD, cpa.CP_TOKEN_MAJOR, w.Hkv, d, 2, k, kh),
                     (cpa.CP_SEQ_TO_HEAD, cpa.CP_TOKEN_MAJOR, w.Hkv, d, 2, v, vh)] + list(extra))
        else:
            kh.view(k.shape).copy_(k)
            vh.view(v.shape).copy_(v)

    def step():
        stage_kv([(cpa.CP_SEQ_TO_HEAD, cpa.CP_TOKEN_MAJOR, w.Hq, d, 2, q, qh)])
        kv = [(kh[i], vh[i]) for i in range(Rl)]
        tr.ring_forward(comm, kern, place, views(qh), kv, views(oh), views(lh))
        reshard([(cpa.CP_HEAD_TO_SEQ, cpa.CP_TOKEN_MAJOR, w.Hq, d, 2, oh, o),
                 (cpa.CP_HEAD_TO_SEQ, cpa.CP_HEAD_MAJOR, w.Hq, 1, 4, lh, lse)])
        if w.backward:
            # K/V again in their owners' buffers (the forward rotated them).
            stage_kv([(cpa.CP_SEQ_TO_HEAD, cpa.CP_TOKEN_MAJOR, w.Hq, d, 2, do, doh)])
            kv = [(kh[i], vh[i]) for i in range(Rl)]
            dkv = tr.ring_backward(comm, kern, place, views(qh), kv, views(oh), views(lh), views(doh), views(dqh))
            dkh = torch.stack([x[0] for x in dkv]) if Rl > 1 else dkv[0][0].unsqueeze(0)
            dvh = torch.stack([x[1] for x in dkv]) if Rl > 1 else dkv[0][1].unsqueeze(0)
            if U > 1:
                reshard([(cpa.CP_HEAD_TO_SEQ, cpa.CP_TOKEN_MAJOR, w.Hq, d, 4, dqh, dq),
                         (cpa.CP_HEAD_TO_SEQ, cpa.CP_TOKEN_MAJOR, w.Hkv, d, 4, dkh, dk),
                         (cpa.CP_HEAD_TO_SEQ, cpa.CP_TOKEN_MAJOR, w.Hkv, d, 4, dvh, dv)])
            else:
                dk.copy_(dkh.view(dk.shape))
                dv.copy_(dvh.view(dv.shape))

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    barrier()
    clocks.start()
    evs = []
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize(dev)
    clock_rec = clocks.stop()
    barrier()
    total_ms = sum(a.elapsed_time(b) for a, b in evs)
    if cpa.cp_get_status(stream) != 0:
        raise RuntimeError("device status set during the timed region")
    # End to end: this process's input slice from pinned host memory, its
    # output slice back, serially around each step.
    in_t = [q, k, v] + ([do] if w.backward else [])
    out_t = [o, lse] + ([dq, dk, dv] if w.backward else [])
    host_in = [t.cpu().pin_memory() for t in in_t]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in out_t]
    e2e_steps = reps_for(total_ms / args.steps, 10)
    barrier()
    ee0, ee1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ee0.record(stream)
    for _ in range(e2e_steps):
        for t, h in zip(in_t, host_in):
            t.copy_(h, non_blocking=True)
        step()
        for t, h in zip(out_t, host_out):
            h.copy_(t, non_blocking=True)
    ee1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = ee0.elapsed_time(ee1) / e2e_steps
    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], dist, dev)
    if rank == 0:
        ms_per_step = total_ms / args.steps
        per_step_launches = ((2 if U > 1 else 0) + Rl * U * (R + 1)
                             + ((3 if U > 1 else 0) + Rl * U * (1 + R) if w.backward else 0))
        peaks, peak_src = load_peaks()
        value = flops_step / (ms_per_step * 1e-3) / 1e12
        cfg = workload_config(w, offsets, args, world, plan.index_map())
        cfg["parallelism"] = (f"one sequence over {world} GPUs: ring transport (NCCL point-to-point), "
                              f"{Rl} ring rank(s) x {U} Ulysses member(s) per GPU" if world > 1 else
                              "ring transport on one GPU: per-step launches, chunks rotated through a loopback")
        peak, plabel = tensor_peak(peaks, peak_src, ms_per_step)
        result = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "strong" if world > 1 else "weak", "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic", "config": cfg,
            "tokens_per_s": round(w.L / (ms_per_step * 1e-3), 1), "useful_flops_per_step": flops_step,
            "gpu_launches": per_step_launches * args.steps,
            "roofline": {"bound": "tensor", "kernel": "attn_fwd_kernel<%d> (one ring step per launch)" % d,
                         "achieved": round(value / world, 2), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(value / world / peak, 4), "peak_source": plabel + ", per GPU",
                         "traffic": None},
            "e2e": {"value": round(flops_step / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in in_t) * world,
                    "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in out_t) * world,
                    "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                    "overlap": "serial per step (copy in, step, copy out) on every GPU"},
            "clocks": clock_rec,
        }
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def cpu_baseline(w, cpu, offsets, flops_full, full=False):
    """The oracle, as it stands, on a bounded seeded sample of the workload,
    with the time a full run would take at the sampled rate; or (full) over
    every query row and head, timed."""
    heads = list(range(w.Hq))
    cores = len(os.sched_getaffinity(0))
    if full:
        import oracle
        per = oracle_rows_per_call(w.L, 256)
        t0 = time.perf_counter()
        for r0 in range(0, w.L, per):
            oracle.attention_rows(cpu["q"], cpu["k"], cpu["v"], rows=np.arange(r0, min(w.L, r0 + per)),
                                  offsets=offsets, heads=heads)
        el = time.perf_counter() - t0
        return {"value": round(flops_full / el / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                "sample": f"full run: all {w.L} query rows x {len(heads)} heads of {w.name} (fp64 numpy, "
                          f"{per} rows per call)",
                "full_run_flops": flops_full, "full_run_s_measured": round(el, 2)}
    rows = oracle_rows_per_call(w.L, 64)
    flops, el, calls = time_oracle(w, cpu, offsets, rows, heads, seed=0, min_seconds=10.0, max_calls=16)
    rate = flops / el
    return {"value": round(rate / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{calls} x {rows} seeded random query rows x {len(heads)} heads of {w.name} "
                      f"(fp64 numpy, {el:.1f} s)",
            "sample_rows_per_s": round(calls * rows / el, 3),
            "full_run_flops": flops_full,
            "full_run_s_extrapolated": round(flops_full / rate, 1),
            "full_run_note": "extrapolated: the full forward's useful FLOPs at the sampled rate, not a measured run"}


def run_reference(args, w, offsets, flops_step, warmup, world):
    """The CPU oracle as the reference arm: each step is a bounded sample (a
    fixed number of seeded random query rows over all heads, fewer rows at
    longer L so that a step stays near a second or two)."""
    import oracle
    cpu = cpu_inputs(w)
    heads = list(range(w.Hq))
    rows = oracle_rows_per_call(w.L, 32)
    rng_seed = 0
    for i in range(warmup):
        time_oracle(w, cpu, offsets, rows, heads, seed=rng_seed + i, min_seconds=0.0, max_calls=1)
    flops = 0
    t = 0.0
    for i in range(args.steps):
        f, el, _ = time_oracle(w, cpu, offsets, rows, heads, seed=1000 + i, min_seconds=0.0, max_calls=1)
        flops += f
        t += el
    value = flops / t / 1e12
    cores = len(os.sched_getaffinity(0))
    sample = f"per step {rows} seeded random query rows x {len(heads)} heads of {w.name} (fp64 numpy oracle)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": warmup,
        "ms_per_step": t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, offsets, args, world,
                                  oracle.ring_positions(w.L, w.ring, w.layout, offsets, args.chunks_per_rank)),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
