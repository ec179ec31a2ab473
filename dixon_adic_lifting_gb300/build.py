"""Builds the C-ABI library ``libexactsolve.so`` in-tree for sm_103a.

Each CUDA translation unit is compiled with
``nvcc -gencode arch=compute_103a,code=sm_103a -lineinfo -O3`` and the host
units with g++; the objects are linked with ``nvcc -shared`` (static CUDA
runtime).  Translation units compile in parallel; objects go to ``_build/``.
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
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libexactsolve.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (CUDA toolkit required to build the library)")
    return cand


def sources():
    cu = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))
    cpp = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cpp"))
    hdr = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hdr.append(os.path.join(ROOT, "include", "es.h"))
    return cu, cpp, hdr


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    cu, cpp, hdr = sources()
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in cu + cpp + hdr + [__file__])


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile every translation unit and link the library; returns its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    cu, cpp, _ = sources()
    inc = ["-I", CSRC, "-I", os.path.join(ROOT, "include")]
    jobs = []
    for f in cu:
        o = os.path.join(BUILD, os.path.basename(f) + ".o")
        cmd = [nvcc, *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC,-O3", *inc, "-c", f, "-o", o]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        jobs.append((cmd, o))
    for f in cpp:
        o = os.path.join(BUILD, os.path.basename(f) + ".o")
        cxx = shutil.which("g++") or "g++"
        jobs.append(([cxx, "-O3", "-std=c++17", "-fPIC", "-pthread", *inc, "-c", f, "-o", o], o))
    outs = []
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        futs = [ex.submit(_run, cmd) for cmd, _ in jobs]
        for fu in futs:
            outs.append(fu.result())
    tmp = LIB + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *[o for _, o in jobs], "-lpthread"])
    os.replace(tmp, LIB)
    if verbose:
        print("\n".join(x for x in outs if x.strip()))
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB)
