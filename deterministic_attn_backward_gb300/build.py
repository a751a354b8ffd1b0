"""Build libdab.so in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in parallel, then linked into a shared
library next to this file.  No CMake; only nvcc and the CUDA headers.
Usage:  python -m deterministic_attn_backward_gb300.build [--verbose-ptxas]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libdab.so")
BUILD_DIR = os.path.join(ROOT, "_build")
SOURCES = ["api.cu", "bwd.cu", "fwd.cu", "aux.cu", "selftest.cu", "dagsim.cpp", "noalloc.cu", "peak.cu", "hostio.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(verbose_ptxas: bool) -> list:
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _deps_mtime() -> float:
    paths = [os.path.join(CSRC, s) for s in os.listdir(CSRC)]
    paths += [os.path.join(INCLUDE, s) for s in os.listdir(INCLUDE)]
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    flags = _flags(verbose_ptxas)
    objs = []
    cmds = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src + ".o")
        objs.append(obj)
        cmds.append([nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj])
    jobs = jobs or min(len(cmds), os.cpu_count() or 1)
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), cmds))
    failed = False
    for cmd, res in zip(cmds, results):
        if res.stdout or res.stderr:
            sys.stderr.write(res.stdout + res.stderr)
        if res.returncode != 0:
            failed = True
            sys.stderr.write(f"FAILED: {' '.join(cmd)}\n")
    if failed:
        raise RuntimeError("nvcc compilation failed")
    tmp = LIB + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lpthread"]
    res = subprocess.run(link, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError("link failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    out = build(force="--force" in sys.argv or "--verbose-ptxas" in sys.argv,
                verbose_ptxas="--verbose-ptxas" in sys.argv)
    print(out)
