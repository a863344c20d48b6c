"""Python binding of libcpattn (include/cp_attn.h): argument marshalling only.

Every function here forwards to the C ABI of the same name; all computation
runs in the library's CUDA kernels.  PyTorch is used only to own device
memory and to name the current stream.  Using this module fails loudly if
the library has not been built (``python -m context_long_sequence_gb300.build``):
the first call raises; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# CPATTN_DEBUG=1 in the environment selects the bounds-checked debug build
# (libcpattn_debug.so, compiled with -DCP_DEBUG) for this process.
DEBUG = os.environ.get("CPATTN_DEBUG", "") not in ("", "0")
LIB_PATH = os.path.join(_HERE, "libcpattn_debug.so" if DEBUG else "libcpattn.so")

# Constants (mirrors include/cp_attn.h).
CP_ATTN_PLAN_VERSION = 1
CP_OK = 0
CP_ERR_INVALID_ARG = -1
CP_ERR_UNSUPPORTED = -2
CP_ERR_ALIGNMENT = -3
CP_ERR_CUDA = -4
CP_ERR_DEVICE_TIMEOUT = -5
CP_ERR_DEVICE_BOUNDS = -6
CP_ERR_WORKSPACE = -7
CP_ERR_ARCH = -8
CP_NOALLOC_SCRATCH_BYTES = 8 << 20
CP_LAYOUT_CONTIGUOUS = 0
CP_LAYOUT_ZIGZAG = 1
CP_LAYOUT_BALANCED = 2
CP_KV_RING = 0
CP_KV_ALLGATHER = 1
CP_SEQ_TO_HEAD = 0
CP_HEAD_TO_SEQ = 1
CP_TOKEN_MAJOR = 0
CP_HEAD_MAJOR = 1
CP_OP_FWD = 0
CP_OP_BWD = 1
CP_OP_BWD_RANK_STATS = 2


CP_RESHARD_MAX_JOBS = 8


class cp_reshard_job_t(ctypes.Structure):
    _fields_ = [
        ("direction", ctypes.c_int32),
        ("tensor_kind", ctypes.c_int32),
        ("H", ctypes.c_int32),
        ("row_elems", ctypes.c_int32),
        ("elem_bytes", ctypes.c_int32),
        ("inp", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
    ]


class cp_plan_desc_t(ctypes.Structure):
    _fields_ = [
        ("version", ctypes.c_int32),
        ("L", ctypes.c_int32),
        ("Hq", ctypes.c_int32),
        ("Hkv", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("ulysses_degree", ctypes.c_int32),
        ("ring_degree", ctypes.c_int32),
        ("layout", ctypes.c_int32),
        ("causal", ctypes.c_int32),
        ("num_docs", ctypes.c_int32),
        ("doc_offsets", ctypes.POINTER(ctypes.c_int32)),
        ("softmax_scale", ctypes.c_float),
        ("emit_partials", ctypes.c_int32),
        ("out_fp32", ctypes.c_int32),
        ("chunks_per_rank", ctypes.c_int32),
        ("kv_exchange", ctypes.c_int32),
    ]


_vp = ctypes.c_void_p
_i = ctypes.c_int
_lib = None


def _L():
    """The loaded library; raises if it has not been built (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{os.path.basename(LIB_PATH)} is not built ({LIB_PATH}); run "
                           "`python -m context_long_sequence_gb300.build` first")
    lib = ctypes.CDLL(LIB_PATH)
    lib.cp_plan_create.argtypes = [ctypes.POINTER(cp_plan_desc_t), ctypes.POINTER(_vp)]
    lib.cp_plan_destroy.argtypes = [_vp]
    lib.cp_plan_destroy.restype = None
    lib.cp_index_map.argtypes = [_vp, ctypes.POINTER(ctypes.c_int32)]
    lib.cp_workspace_size.argtypes = [_vp, _i, ctypes.POINTER(ctypes.c_size_t)]
    lib.ulysses_reshard.argtypes = [_vp, _i, _i, _i, _i, _i, _vp, _vp, _vp]
    lib.ulysses_reshard_batch.argtypes = [_vp, _i, ctypes.POINTER(cp_reshard_job_t), _vp]
    lib.cp_attn_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.cp_attn_fwd_local.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.cp_attn_fwd_rank.argtypes = [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.cp_attn_fwd_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.cp_attn_bwd.argtypes = [_vp] + [_vp] * 9 + [_vp, ctypes.c_size_t, _vp]
    lib.cp_attn_fwd_step.argtypes = [_vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.cp_attn_bwd_delta.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp]
    lib.cp_attn_bwd_step.argtypes = [_vp, _i, _i] + [_vp] * 8 + [_vp]
    lib.cp_merge_lse.argtypes = [_i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp]
    lib.cp_get_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_int32)]
    lib.cp_selftest_wait_timeout.argtypes = [ctypes.c_int32, ctypes.POINTER(ctypes.c_int32), _vp]
    lib.cp_selftest_bounds.argtypes = [ctypes.c_int32, ctypes.POINTER(ctypes.c_int32), _vp]
    lib.cp_get_status_detail.argtypes = [_vp, ctypes.POINTER(ctypes.c_int32)]
    lib.cp_tile_classes.argtypes = [_vp, ctypes.POINTER(ctypes.c_int32), ctypes.c_int64,
                                    ctypes.POINTER(ctypes.c_int64), _vp]
    lib.cp_debug_build.argtypes = []
    lib.cp_measure_rates.argtypes = [ctypes.POINTER(ctypes.c_double), _vp]
    lib.cp_measure_barrier_check.argtypes = [ctypes.POINTER(ctypes.c_double), _vp]
    lib.cp_strerror.argtypes = [_i]
    lib.cp_strerror.restype = ctypes.c_char_p
    _lib = lib
    return lib


EXPORTED = ["cp_plan_create", "cp_plan_destroy", "cp_index_map", "cp_workspace_size", "ulysses_reshard",
            "ulysses_reshard_batch",
            "cp_attn_fwd", "cp_attn_fwd_local", "cp_attn_fwd_rank", "cp_attn_fwd_noalloc", "cp_attn_bwd",
            "cp_attn_fwd_step", "cp_attn_bwd_delta", "cp_attn_bwd_step",
            "cp_merge_lse", "cp_get_status", "cp_get_status_detail", "cp_debug_build", "cp_strerror",
            "cp_selftest_wait_timeout", "cp_selftest_bounds", "cp_tile_classes", "cp_measure_rates", "cp_measure_barrier_check"]


class CPError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {cp_strerror(code)} ({code})")


def cp_strerror(code: int) -> str:
    return _L().cp_strerror(int(code)).decode()


def _check(rc: int, where: str):
    if rc != CP_OK:
        raise CPError(rc, where)


def _ptr(x):
    """Device address of a tensor (or an int address); None -> NULL."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """Owns a cp_plan_t (cp_plan_create / cp_plan_destroy)."""

    def __init__(self, L, Hq, Hkv, d, ulysses_degree=1, ring_degree=1, layout=CP_LAYOUT_CONTIGUOUS,
                 doc_offsets=None, softmax_scale=0.0, emit_partials=False, causal=True, out_fp32=False,
                 chunks_per_rank=8, kv_exchange=CP_KV_RING):
        self._h = None
        desc = cp_plan_desc_t()
        desc.version = CP_ATTN_PLAN_VERSION
        desc.L, desc.Hq, desc.Hkv, desc.d = int(L), int(Hq), int(Hkv), int(d)
        desc.ulysses_degree, desc.ring_degree = int(ulysses_degree), int(ring_degree)
        desc.layout = int(layout)
        desc.causal = 1 if causal else 0
        self._offsets = None
        if doc_offsets is not None and len(doc_offsets) > 2:
            self._offsets = (ctypes.c_int32 * len(doc_offsets))(*[int(x) for x in doc_offsets])
            desc.num_docs = len(doc_offsets) - 1
            desc.doc_offsets = ctypes.cast(self._offsets, ctypes.POINTER(ctypes.c_int32))
        else:
            desc.num_docs = 0
            desc.doc_offsets = None
        desc.softmax_scale = float(softmax_scale)
        desc.emit_partials = 1 if emit_partials else 0
        desc.out_fp32 = 1 if out_fp32 else 0
        desc.chunks_per_rank = int(chunks_per_rank)
        desc.kv_exchange = int(kv_exchange)
        h = _vp()
        _check(_L().cp_plan_create(ctypes.byref(desc), ctypes.byref(h)), "cp_plan_create")
        self._h = h
        self.L, self.Hq, self.Hkv, self.d = desc.L, desc.Hq, desc.Hkv, desc.d
        self.U, self.R = desc.ulysses_degree, desc.ring_degree
        self.P = self.U * self.R
        self.n = self.L // self.P
        self.layout = desc.layout
        self.chunks_per_rank = desc.chunks_per_rank
        self.kv_exchange = desc.kv_exchange
        self.emit_partials = bool(emit_partials)
        self.out_fp32 = bool(out_fp32)

    @property
    def o_dtype(self):
        import torch
        return torch.float32 if self.out_fp32 else torch.bfloat16

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h is not None:
            _L().cp_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def index_map(self) -> np.ndarray:
        out = np.empty(self.L, dtype=np.int32)
        _check(_L().cp_index_map(self._h, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))), "cp_index_map")
        return out

    def workspace_size(self, op=CP_OP_FWD) -> int:
        n = ctypes.c_size_t()
        _check(_L().cp_workspace_size(self._h, int(op), ctypes.byref(n)), "cp_workspace_size")
        return n.value


def ulysses_reshard(plan: Plan, direction, tensor_kind, H, row_elems, elem_bytes, inp, out, stream=None):
    _check(_L().ulysses_reshard(plan.handle, int(direction), int(tensor_kind), int(H), int(row_elems),
                                int(elem_bytes), _ptr(inp), _ptr(out), _stream(stream)), "ulysses_reshard")


def ulysses_reshard_batch(plan: Plan, jobs, stream=None):
    """jobs: sequence of (direction, tensor_kind, H, row_elems, elem_bytes, inp, out)."""
    arr = (cp_reshard_job_t * max(1, len(jobs)))()
    for i, (direction, kind, H, row_elems, elem_bytes, inp, out) in enumerate(jobs):
        arr[i] = cp_reshard_job_t(int(direction), int(kind), int(H), int(row_elems), int(elem_bytes),
                                  _ptr(inp), _ptr(out))
    _check(_L().ulysses_reshard_batch(plan.handle, len(jobs), arr, _stream(stream)), "ulysses_reshard_batch")


def cp_attn_fwd(plan: Plan, q, k, v, o, lse, workspace=None, workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_L().cp_attn_fwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace),
                            int(workspace_bytes), _stream(stream)), "cp_attn_fwd")


def cp_attn_fwd_rank(plan: Plan, rank, q, k, v, o, lse, stream=None):
    _check(_L().cp_attn_fwd_rank(plan.handle, int(rank), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                 _stream(stream)), "cp_attn_fwd_rank")


def cp_attn_fwd_local(plan: Plan, q, k, v, o, lse, stream=None):
    _check(_L().cp_attn_fwd_local(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _stream(stream)),
           "cp_attn_fwd_local")


def cp_attn_fwd_noalloc(plan: Plan, q, k, v, o, lse, stream=None):
    """cp_attn_fwd for an emit-partials plan, with the partials kept in the
    library's static device scratch instead of an allocated workspace."""
    _check(_L().cp_attn_fwd_noalloc(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _stream(stream)),
           "cp_attn_fwd_noalloc")


def cp_attn_bwd(plan: Plan, q, k, v, o, lse, dO, dq, dk, dv, workspace=None, workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_L().cp_attn_bwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                            _ptr(dk), _ptr(dv), _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "cp_attn_bwd")


def cp_attn_fwd_step(plan: Plan, rank, step, q_rank, k_chunk, v_chunk, o_part, lse_part, stream=None):
    _check(_L().cp_attn_fwd_step(plan.handle, int(rank), int(step), _ptr(q_rank), _ptr(k_chunk), _ptr(v_chunk),
                                 _ptr(o_part), _ptr(lse_part), _stream(stream)), "cp_attn_fwd_step")


def cp_attn_bwd_delta(plan: Plan, o_rank, do_rank, lse_rank, stats_rank, stream=None):
    _check(_L().cp_attn_bwd_delta(plan.handle, _ptr(o_rank), _ptr(do_rank), _ptr(lse_rank), _ptr(stats_rank),
                                  _stream(stream)), "cp_attn_bwd_delta")


def cp_attn_bwd_step(plan: Plan, rank, step, q_rank, do_rank, stats_rank, k_chunk, v_chunk, dq_rank, dk_chunk,
                     dv_chunk, stream=None):
    _check(_L().cp_attn_bwd_step(plan.handle, int(rank), int(step), _ptr(q_rank), _ptr(do_rank), _ptr(stats_rank),
                                 _ptr(k_chunk), _ptr(v_chunk), _ptr(dq_rank), _ptr(dk_chunk), _ptr(dv_chunk),
                                 _stream(stream)), "cp_attn_bwd_step")


def cp_merge_lse(n_parts, rows, H, d, o_parts, lse_parts, o_out, lse_out, stream=None):
    _check(_L().cp_merge_lse(int(n_parts), int(rows), int(H), int(d), _ptr(o_parts), _ptr(lse_parts),
                             _ptr(o_out), _ptr(lse_out), _stream(stream)), "cp_merge_lse")


def cp_selftest_wait_timeout(limit_us, stream=None):
    """Run the bounded-wait self-test; returns (timed_out, left_on_abort, wait_us)."""
    out = (ctypes.c_int32 * 3)()
    _check(_L().cp_selftest_wait_timeout(int(limit_us), out, _stream(stream)), "cp_selftest_wait_timeout")
    return int(out[0]), int(out[1]), int(out[2])


def cp_tile_classes(plan, stream=None) -> np.ndarray:
    """The forward's tile-class table of `plan`: int32 [n][8] rows
    {a, q0, len, step, kpos0, klen, class0, class1} (see include/cp_attn.h)."""
    n = ctypes.c_int64()
    _check(_L().cp_tile_classes(plan.handle, None, 0, ctypes.byref(n), _stream(stream)), "cp_tile_classes")
    out = np.zeros((max(n.value, 1), 8), dtype=np.int32)
    _check(_L().cp_tile_classes(plan.handle, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n.value,
                                ctypes.byref(n), _stream(stream)), "cp_tile_classes")
    return out[:n.value]


def cp_selftest_bounds(block, stream=None) -> int:
    """Run the bounds-record self-test in block `block`; returns the source
    line the kernel recorded (read the record with cp_get_status_detail)."""
    line = ctypes.c_int32()
    _check(_L().cp_selftest_bounds(int(block), ctypes.byref(line), _stream(stream)), "cp_selftest_bounds")
    return line.value


def cp_get_status_detail(stream=None):
    """Read and clear the device status record: (code, block, line, file id)."""
    out = (ctypes.c_int32 * 4)()
    _check(_L().cp_get_status_detail(_stream(stream), out), "cp_get_status_detail")
    return tuple(int(x) for x in out)


def cp_measure_rates(stream=None):
    """(ex2 results per SM clock, SM clocks per M128 N128 K16 bf16 MMA)."""
    out = (ctypes.c_double * 2)()
    _check(_L().cp_measure_rates(out, _stream(stream)), "cp_measure_rates")
    return float(out[0]), float(out[1])


def cp_measure_barrier_check(stream=None) -> float:
    """SM clocks per warp-wide check of a completed mbarrier phase."""
    out = ctypes.c_double(0.0)
    _check(_L().cp_measure_barrier_check(ctypes.byref(out), _stream(stream)), "cp_measure_barrier_check")
    return float(out.value)


def cp_debug_build() -> bool:
    """True when the loaded library is the -DCP_DEBUG build."""
    return bool(_L().cp_debug_build())


def cp_get_status(stream=None) -> int:
    code = ctypes.c_int32()
    _check(_L().cp_get_status(_stream(stream), ctypes.byref(code)), "cp_get_status")
    return code.value


def alloc_workspace(plan: Plan, op=CP_OP_FWD, device="cuda"):
    """A device byte buffer of cp_workspace_size() bytes (None when zero)."""
    import torch
    n = plan.workspace_size(op)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None
