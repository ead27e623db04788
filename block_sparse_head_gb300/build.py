"""In-tree build of libbsa.so for sm_103a (nvcc, no cmake).

Each translation unit compiles to ``_build/<name>.o`` in parallel; the shared library
is linked next to this file.  Objects are rebuilt when a source or header is newer.
Usage: ``python -m block_sparse_head_gb300.build [--force] [-v]``.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libbsa.so")

SOURCES = [
    "bsa_host.cpp",
    "bsa_selftest.cu",
    "bsa_noalloc.cu",
    "bsa_topk.cu",
] + [f"bsa_fwd_q{qb}_k{kb}_d{d}.cu" for qb, kb in ((64, 64), (128, 128), (64, 128), (128, 64))
     for d in (64, 128)] + [f"bsa_bwd_b{b}_d{d}.cu" for b in (64, 128) for d in (64, 128)]
HEADERS = ["bsa_internal.h", "bsa_ptx.cuh", "bsa_fwd_kernel.cuh", "bsa_bwd_kernel.cuh",
           "bsa_topk_kernel.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbsa.so")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile every kernel and the host library; returns the path of libbsa.so."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "bsa.h")]
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        objs.append(o)
        if force or _stale(o, [s] + headers):
            cmd = [nvcc] + FLAGS + (["-Xptxas", "-v"] if ptxas_verbose else []) + ["-c", s, "-o", o]
            jobs.append((src, cmd))

    def run(job):
        src, cmd = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, cmd, r

    failed = []
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for src, cmd, r in ex.map(run, jobs):
                if verbose or ptxas_verbose or r.returncode != 0:
                    sys.stderr.write(f"[bsa build] {src}\n{r.stdout}{r.stderr}")
                if r.returncode != 0:
                    failed.append(src)
    if failed:
        raise RuntimeError(f"libbsa build failed for {failed}")
    if force or jobs or _stale(LIB, objs):
        cmd = [nvcc] + ARCH + ["-shared", "-o", LIB] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"libbsa link failed:\n{r.stdout}{r.stderr}")
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv,
          ptxas_verbose="--ptxas" in sys.argv)
    print(LIB)
