"""Build libdash.so in-tree with nvcc (sm_103a only).

Usage: ``python -m tile_scheduling_persistent_gb300.build [-v]`` or
``build()`` from Python.  Objects go to ``_build/`` at the repository root;
the shared library lands next to this file.  Translation units compile in
parallel; no cmake.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "libdash.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

CUDA_SOURCES = ["dash_bwd.cu", "dash_fwd.cu", "dash_aux.cu", "dash_probe.cu", "dash_api.cu", "dash_noalloc.cu"]
CXX_SOURCES = ["dash_sim.cpp"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed: %s\n%s" % (" ".join(cmd), r.stdout))
    return r.stdout


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    nvcc = _nvcc()
    bdir = os.path.join(ROOT, "_build")
    os.makedirs(bdir, exist_ok=True)
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    jobs = []
    for src in CUDA_SOURCES:
        obj = os.path.join(bdir, src + ".o")
        cmd = [nvcc, *ARCH, "-lineinfo", *common, "--expt-relaxed-constexpr", "-c",
               os.path.join(CSRC, src), "-o", obj]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        jobs.append((cmd, obj))
    for src in CXX_SOURCES:
        obj = os.path.join(bdir, src + ".o")
        cmd = [nvcc, "-x", "c++", *common, "-c", os.path.join(CSRC, src), "-o", obj]
        jobs.append((cmd, obj))
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        logs = list(ex.map(lambda j: _run(j[0], verbose), jobs))
    if ptxas_info:
        for log in logs:
            if log.strip():
                print(log)
    tmp = OUT + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *[o for _, o in jobs], "-lpthread", "-ldl", "-lrt"], verbose)
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv))
