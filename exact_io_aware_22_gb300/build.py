"""Builds the sm_103a CUDA library ``_build/libfa_gb300.so`` in-tree with nvcc.

Each translation unit compiles in parallel; ``-Xptxas -v`` register/spill
reports go to ``_build/ptxas_<unit>.log``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libfa_gb300.so")
UNITS = ["fa_api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_bwd128.cu", "fa_bwd64.cu", "fa_decode.cu",
         "fa_fwd8.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-v", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; set NVCC or put the CUDA toolkit on PATH")
    return cand


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every unit for sm_103a and link the shared library; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(ROOT, "include", "fa.h"))
    objs = []
    jobs = []
    for u in UNITS:
        src = os.path.join(CSRC, u)
        obj = os.path.join(BUILD, u.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            log = os.path.join(BUILD, "ptxas_" + u.replace(".cu", ".log"))
            jobs.append(([nvcc] + ARCH + FLAGS + ["-c", src, "-o", obj], log))

    def run(job):
        cmd, log = job
        p = subprocess.run(cmd, capture_output=True, text=True)
        with open(log, "w") as f:
            f.write(p.stdout + p.stderr)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed ({' '.join(cmd[-3:])}):\n{p.stderr[-4000:]}")
        if verbose:
            print(p.stderr)

    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
