"""Host-side checks of the C ABI that need no GPU: every symbol the header
declares is exported, plan validation returns the documented codes, the
index map matches the oracle's, and workspace sizes follow their formula."""
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def cpa():
    lib = os.path.join(ROOT, "context_long_sequence_gb300", "libcpattn.so")
    if not os.path.exists(lib):
        from context_long_sequence_gb300 import build as b
        b.build()
    import context_long_sequence_gb300 as m
    return m


def declared_functions():
    src = open(os.path.join(ROOT, "include", "cp_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(\w+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_header_symbols_exported(cpa):
    names = declared_functions()
    assert "cp_attn_fwd" in names and "ulysses_reshard" in names and "cp_merge_lse" in names
    out = subprocess.run(["nm", "-D", "--defined-only", cpa.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    assert sorted(names) == sorted(cpa.EXPORTED)
    for n in names:
        getattr(cpa._L(), n)


def test_debug_library_exports_and_flag(cpa):
    """The -DCP_DEBUG variant exports the same symbols and says it is the
    debug build; the release library says it is not (host-only calls)."""
    import ctypes
    dbg = os.path.join(ROOT, "context_long_sequence_gb300", "libcpattn_debug.so")
    if not os.path.exists(dbg):
        from context_long_sequence_gb300 import build as b
        b.build()
    out = subprocess.run(["nm", "-D", "--defined-only", dbg], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    assert ctypes.CDLL(dbg).cp_debug_build() == 1
    assert cpa._L().cp_debug_build() == (1 if cpa.DEBUG else 0)


def test_reshard_batch_argument_checks(cpa):
    """ulysses_reshard_batch rejects bad job counts, misaligned pointers and
    overlapping buffers before touching the device (fake addresses)."""
    p = cpa.Plan(1024, 8, 4, 64, ulysses_degree=4, ring_degree=2, layout=1)
    nbytes = 1024 * 8 * 64 * 2
    base = 1 << 36
    job = lambda i, o: (cpa.CP_SEQ_TO_HEAD, cpa.CP_TOKEN_MAJOR, 8, 64, 2, i, o)
    L = cpa._L()

    def call(jobs, n=None):
        arr = (cpa.cp_reshard_job_t * max(1, len(jobs)))()
        for i, j in enumerate(jobs):
            arr[i] = cpa.cp_reshard_job_t(*j[:5], j[5], j[6])
        return L.ulysses_reshard_batch(p.handle, len(jobs) if n is None else n, arr, None)
    a, b, c, d = base, base + 4 * nbytes, base + 8 * nbytes, base + 12 * nbytes
    assert call([job(a, b)], n=0) == cpa.CP_ERR_INVALID_ARG
    assert call([job(a, b)] * 9) == cpa.CP_ERR_INVALID_ARG
    assert call([job(a + 8, b)]) == cpa.CP_ERR_ALIGNMENT
    assert call([job(a, b), job(c, b + 256)]) == cpa.CP_ERR_INVALID_ARG      # two outputs overlap
    assert call([job(a, b), job(b + 512, d)]) == cpa.CP_ERR_INVALID_ARG      # an input inside an output
    assert call([job(a, a + 256)]) == cpa.CP_ERR_INVALID_ARG                 # in and out overlap
    assert call([(cpa.CP_SEQ_TO_HEAD, cpa.CP_TOKEN_MAJOR, 6, 64, 2, a, b)]) == cpa.CP_ERR_INVALID_ARG  # U does not divide H
    assert L.ulysses_reshard_batch(p.handle, 1, None, None) == cpa.CP_ERR_INVALID_ARG


def test_measure_rates_argument_check(cpa):
    assert cpa._L().cp_measure_rates(None, None) == cpa.CP_ERR_INVALID_ARG
    assert cpa._L().cp_measure_barrier_check(None, None) == cpa.CP_ERR_INVALID_ARG


def test_tile_classes_argument_checks(cpa):
    import ctypes
    p = cpa.Plan(512, 4, 2, 64, ring_degree=2, layout=1)
    n = ctypes.c_int64()
    assert cpa._L().cp_tile_classes(p.handle, None, 0, None, None) == cpa.CP_ERR_INVALID_ARG
    assert cpa._L().cp_tile_classes(p.handle, None, -1, ctypes.byref(n), None) == cpa.CP_ERR_INVALID_ARG
    assert cpa._L().cp_tile_classes(p.handle, None, 5, ctypes.byref(n), None) == cpa.CP_ERR_INVALID_ARG
    assert cpa._L().cp_tile_classes(None, None, 0, ctypes.byref(n), None) == cpa.CP_ERR_INVALID_ARG


@pytest.mark.parametrize("L,R,U,layout", [(64, 4, 1, 0), (64, 4, 1, 1), (96, 3, 2, 1), (128, 2, 4, 1),
                                          (1024, 8, 1, 1), (48, 1, 1, 1), (2048, 8, 4, 1)])
def test_index_map_matches_oracle(cpa, L, R, U, layout):
    import oracle
    p = cpa.Plan(L, 8, 4, 64, ulysses_degree=U, ring_degree=R, layout=layout)
    assert np.array_equal(p.index_map(), oracle.ring_positions(L, R, layout))


@pytest.mark.parametrize("L,R,U,m,docs", [
    (24, 2, 1, 3, [0, 10, 24]), (16, 2, 1, 2, [0, 3, 16]), (12, 3, 1, 1, None), (65536, 8, 1, 2, None),
    (4096, 4, 2, 4, [0, 100, 2000, 4096]), (1000, 5, 1, 4, [0, 1, 2, 999, 1000]), (131072, 16, 1, 8, "packed")])
def test_balanced_index_map_matches_oracle(cpa, L, R, U, m, docs):
    """The plan's work-balanced chunk assignment (C++) equals the oracle's,
    bit for bit, including the packed-document workload's seeded documents."""
    import oracle
    import workloads
    if docs == "packed":
        docs = workloads.workload_doc_offsets(workloads.WORKLOADS[3])
    p = cpa.Plan(L, 8, 4, 64, ulysses_degree=U, ring_degree=R, layout=cpa.CP_LAYOUT_BALANCED, doc_offsets=docs,
                 chunks_per_rank=m)
    assert np.array_equal(p.index_map(), oracle.ring_positions(L, R, oracle.LAYOUT_BALANCED, docs, m))


@pytest.mark.parametrize("kw,code", [
    (dict(L=100, Hq=8, Hkv=4, d=64, ring_degree=3), -1),                 # R does not divide L
    (dict(L=96, Hq=8, Hkv=3, d=64), -1),                                 # Hkv does not divide Hq
    (dict(L=96, Hq=8, Hkv=4, d=96), -2),                                 # head dim not built
    (dict(L=96, Hq=8, Hkv=4, d=64, ulysses_degree=8), -2),               # U must divide Hkv
    (dict(L=96, Hq=8, Hkv=4, d=64, causal=False), -2),
    (dict(L=96, Hq=8, Hkv=4, d=64, ulysses_degree=2, emit_partials=True), -2),
    (dict(L=96, Hq=8, Hkv=4, d=64, doc_offsets=[0, 50, 40, 96]), -1),    # not increasing
    (dict(L=96, Hq=8, Hkv=4, d=64, doc_offsets=[0, 50, 95]), -1),        # does not end at L
    (dict(L=90, Hq=8, Hkv=4, d=64, ring_degree=4, layout=1), -1),        # 2R does not divide L
    (dict(L=96, Hq=8, Hkv=4, d=64, ulysses_degree=4, ring_degree=5), -1),
    (dict(L=96, Hq=8, Hkv=4, d=64, ring_degree=2, layout=2, chunks_per_rank=0), -1),   # balanced needs m >= 1
    (dict(L=96, Hq=8, Hkv=4, d=64, ring_degree=2, layout=2, chunks_per_rank=5), -1),   # m*R does not divide L
    (dict(L=96, Hq=8, Hkv=4, d=64, layout=3), -1),                                    # unknown layout
    (dict(L=96, Hq=8, Hkv=4, d=64, kv_exchange=2), -1),                               # unknown KV exchange
    (dict(L=96, Hq=8, Hkv=4, d=64, ulysses_degree=2, kv_exchange=1), -2),             # all-gather is U == 1
    (dict(L=96, Hq=8, Hkv=4, d=64, ring_degree=2, emit_partials=True, kv_exchange=1), -2),
])
def test_plan_validation(cpa, kw, code):
    with pytest.raises(cpa.CPError) as e:
        cpa.Plan(**kw)
    assert e.value.code == code


def test_workspace_sizes(cpa):
    def al(x):
        return (x + 255) // 256 * 256
    p = cpa.Plan(16384, 32, 8, 128, ulysses_degree=4)
    L = 16384
    assert p.workspace_size(cpa.CP_OP_FWD) == 0   # the Ulysses exchanges are the kernel's addressing
    # Row statistics (-LSE*log2e, -D; chunks already multiples of 128).
    assert p.workspace_size(cpa.CP_OP_BWD) == al(L * 32 * 4) * 2   # row statistics only: no head-sharded copies
    assert p.workspace_size(cpa.CP_OP_BWD_RANK_STATS) == 2 * 8 * 16384 * 4  # T = L/R = 16384 slots, 8 heads
    p = cpa.Plan(16384, 32, 8, 128, ring_degree=4)
    assert p.workspace_size(cpa.CP_OP_BWD) == al(L * 32 * 4) * 2
    # Ragged chunks pad to 128 slots: T = 500, two chunks of 250 -> 2 x 256.
    p = cpa.Plan(1000, 4, 2, 64, ring_degree=2, layout=1)
    assert p.workspace_size(cpa.CP_OP_BWD_RANK_STATS) == 2 * 4 * 512 * 4
    assert p.workspace_size(cpa.CP_OP_BWD) == al(2 * 4 * 512 * 4) * 2
    p = cpa.Plan(1024, 4, 4, 64, ring_degree=4, emit_partials=True)
    assert p.workspace_size(cpa.CP_OP_FWD) == al(4 * 1024 * 4 * 64 * 4) + al(4 * 1024 * 4 * 4)
    p = cpa.Plan(1024, 4, 4, 64, ring_degree=4)
    assert p.workspace_size(cpa.CP_OP_FWD) == 0
    p = cpa.Plan(1000, 4, 2, 64, ring_degree=4, layout=1, kv_exchange=cpa.CP_KV_ALLGATHER)
    assert p.workspace_size(cpa.CP_OP_FWD) == 2 * al(1000 * 2 * 64 * 2)   # gathered K and V


def test_fwd_rank_rejects_bad_rank(cpa):
    p = cpa.Plan(1024, 4, 2, 64, ring_degree=4)
    fake = 256  # aligned, never dereferenced: the rank check comes first
    for r in (-1, 4):
        assert cpa._L().cp_attn_fwd_rank(p.handle, r, fake, fake, fake, fake, fake, None) == cpa.CP_ERR_INVALID_ARG


def test_strerror(cpa):
    assert cpa.cp_strerror(0) == "ok"
    assert "align" in cpa.cp_strerror(cpa.CP_ERR_ALIGNMENT)
    assert cpa.cp_strerror(12345) == "unknown error"
