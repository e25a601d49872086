"""Build libmoedecode.so in-tree with nvcc for sm_103a.

Each .cu file compiles to an object in parallel; the objects link into one
shared library next to this file. Rebuilds only what changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmoedecode.so")
ARCH = os.environ.get("MOE_DECODE_ARCH", "103a")

SOURCES = ["api.cu", "gemv.cu", "umma.cu", "router.cu", "misc.cu", "noalloc.cu", "gemv_moe.cu", "route_shared.cu"]
HEADERS = ["common.cuh", "internal.h"]
PUBLIC = os.path.join(ROOT, "include", "moe_decode.h")


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def flags() -> list:
    # MOE_DECODE_NVCC_EXTRA: extra nvcc flags (e.g. -DDEC_ENGINE_KSUB_SINGLE=4) for tuning builds.
    extra = os.environ.get("MOE_DECODE_NVCC_EXTRA", "").split()
    return ["-O3", "-std=c++17", f"-gencode=arch=compute_{ARCH},code=sm_{ARCH}", "-lineinfo",
            "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")] + extra


def _mtime(p: str) -> float:
    return os.path.getmtime(p) if os.path.exists(p) else -1.0


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    stamp = os.path.join(BUILD, "flags.txt")
    want = " ".join(flags())
    if not os.path.exists(stamp) or open(stamp).read() != want:
        for f in os.listdir(BUILD):
            if f.endswith(".o"):
                os.remove(os.path.join(BUILD, f))
        with open(stamp, "w") as fh:
            fh.write(want)
    deps = [os.path.join(CSRC, h) for h in HEADERS] + [PUBLIC]
    dep_time = max(_mtime(d) for d in deps)
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if ptxas_info or _mtime(o) < max(_mtime(s), dep_time):
            cmd = [nvcc()] + flags() + (["-Xptxas", "-v"] if ptxas_info else []) + ["-c", s, "-o", o]
            jobs.append(cmd)
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs))
        for cmd, r in zip(jobs, results):
            if verbose or ptxas_info or r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    if jobs or _mtime(LIB) < max(_mtime(o) for o in objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc(), "-shared", f"-gencode=arch=compute_{ARCH},code=sm_{ARCH}", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB)
