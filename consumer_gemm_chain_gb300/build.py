"""Builds the C-ABI shared libraries in-tree with nvcc for sm_103a.

Two builds of the same sources and ABI are made in parallel:
``_lib/libcs_chain.so`` (everything) and ``_lib/libcs_chain_nomc.so``, the
replica build compiled with ``-DCS_NO_CLUSTER_MULTICAST``: it contains no TMA
cluster-multicast load (no 512-row tiles), and it is the one the binding loads
in a process that shares a node with other GPUs' ranks."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libcs_chain.so")
LIB_NOMC = os.path.join(LIBDIR, "libcs_chain_nomc.so")
# (library, extra nvcc defines)
VARIANTS = ((LIB, []), (LIB_NOMC, ["-DCS_NO_CLUSTER_MULTICAST"]))
SOURCES = ["cs_chain.cu", "cs_tune.cpp"]
DEPS = ["cs_chain.cu", "cs_kernel.cuh", "cs_ptx.cuh", "cs_sched.cuh", "cs_tune.cpp", "cs_tune.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, d) for d in DEPS] + [os.path.join(ROOT, "include", "cs_chain.h")]
    return any(os.path.exists(d) and os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile both libraries where any source is newer (in parallel); returns the
    path of the full one."""
    todo = [(lib, defs) for lib, defs in VARIANTS if force or _stale(lib)]
    if not todo:
        return LIB
    os.makedirs(LIBDIR, exist_ok=True)
    procs = []
    for lib, defs in todo:
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [_nvcc(), *ARCH, *defs, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-shared",
               "-I", os.path.join(ROOT, "include"), "-o", tmp] + [os.path.join(CSRC, s) for s in SOURCES]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
            print(" ".join(cmd), file=sys.stderr)
        procs.append((lib, tmp, cmd, subprocess.Popen(cmd)))
    failed = [cmd for _, _, cmd, pr in procs if pr.wait() != 0]
    if failed:
        raise subprocess.CalledProcessError(1, failed[0])
    for lib, tmp, _, _ in procs:
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
