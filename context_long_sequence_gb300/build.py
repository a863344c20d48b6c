"""Build libcpattn.so in-tree with nvcc for sm_103a (no cmake, no torch).

Each .cu is compiled to an object in parallel, then linked into one shared
library next to this file.  The same sources compiled with -DCP_DEBUG give
libcpattn_debug.so, whose kernels check every work item, global index and
TMA coordinate and record failures in the device status words (see
cp_get_status_detail in include/cp_attn.h).  Both variants compile at once.
Usage: ``python -m context_long_sequence_gb300.build [--release-only]``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libcpattn.so")
LIB_DEBUG = os.path.join(PKG, "libcpattn_debug.so")
BUILD_DIR = os.path.join(PKG, "_build")
SOURCES = ["cp_attn.cu", "attn_fwd.cu", "attn_bwd.cu", "reshard.cu", "merge.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def flags(extra=()):
    return [*ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
            "--expt-relaxed-constexpr", *extra]


def _start(variant_dir: str, extra, verbose: bool):
    os.makedirs(variant_dir, exist_ok=True)
    cc = nvcc()
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(variant_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [cc, *flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd))
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    return procs, objs


def _finish(procs, objs, lib: str, verbose: bool) -> str:
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append(f"--- {src}\n{out}")
        elif verbose and out.strip():
            print(out)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = lib + ".tmp"
    link = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-ldl"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, lib)
    return lib


def build(verbose: bool = False, extra=(), debug: bool = True) -> str:
    """Compile the release library (and, with `debug`, the -DCP_DEBUG one
    alongside it, in parallel).  Returns the release library's path."""
    rel = _start(BUILD_DIR, extra, verbose)
    dbg = _start(os.path.join(BUILD_DIR, "debug"), [*extra, "-DCP_DEBUG"], verbose) if debug else None
    _finish(*rel, LIB, verbose)
    if dbg is not None:
        _finish(*dbg, LIB_DEBUG, verbose)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, extra=["-Xptxas", "-v"] if "--ptxas" in sys.argv else [],
                debug="--release-only" not in sys.argv))
