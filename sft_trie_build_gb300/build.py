"""Builds libstp.so in-tree: nvcc for the CUDA sources (sm_103a only), g++
for the host packer, compiled in parallel and linked with the static CUDA
runtime.  No cmake; a couple of minutes at most."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libstp.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "--expt-relaxed-constexpr", "-Xptxas", "-v", "-I", os.path.join(ROOT, "include")]
CXX_FLAGS = ["-O2", "-fPIC", "-std=c++17", "-Wall", "-pthread", "-I", os.path.join(ROOT, "include")]


def _nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def sources():
    cu = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    cpp = sorted(f for f in os.listdir(CSRC) if f.endswith(".cpp"))
    return cu, cpp


def _run(cmd, log):
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + p.stdout)
    if p.returncode != 0:
        raise RuntimeError(f"build step failed ({p.returncode}): {' '.join(cmd)}\n{p.stdout[-4000:]}")
    return p.stdout


def build(verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    cu, cpp = sources()
    jobs = []
    objs = []
    for f in cu:
        o = os.path.join(BUILD, f + ".o")
        objs.append(o)
        jobs.append(([nvcc] + NVCC_FLAGS + ["-c", os.path.join(CSRC, f), "-o", o],
                     os.path.join(BUILD, f + ".log")))
    cxx = os.environ.get("CXX", "g++")
    for f in cpp:
        o = os.path.join(BUILD, f + ".o")
        objs.append(o)
        jobs.append(([cxx] + CXX_FLAGS + ["-c", os.path.join(CSRC, f), "-o", o],
                     os.path.join(BUILD, f + ".log")))
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        outs = list(ex.map(lambda j: _run(*j), jobs))
    if verbose:
        for (cmd, _), out in zip(jobs, outs):
            if out.strip():
                print(out)
    tmp = LIB + ".tmp"
    _run([nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs + ["-lpthread", "-ldl", "-lrt"],
         os.path.join(BUILD, "link.log"))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
