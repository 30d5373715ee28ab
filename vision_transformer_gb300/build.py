"""Builds libsv.so (the CUDA library) in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel to ``_build/*.o``; the shared
library links them with the static CUDA runtime. Host code uses portable
flags only (the library is built on x86-64 and on aarch64 hosts).
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
LIB = os.path.join(HERE, "libsv.so")
SOURCES = ["api.cu", "gemm_tc.cu", "attention.cu", "elementwise.cu", "map_static.cu"]
HEADERS = ["ptx.cuh", "sv_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps():
    return ([os.path.join(CSRC, h) for h in HEADERS]
            + [os.path.join(ROOT, "include", "sv.h"), os.path.join(ROOT, "synth", "synth.h")])


def _stale(out: str, inputs) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(p) > t for p in inputs)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    flags = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"] + ARCH
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + _deps()):
            jobs.append([cc] + flags + ["-c", s, "-o", o] + (["-Xptxas", "-v"] if verbose else []))
    synth_src = os.path.join(ROOT, "synth", "synth.cpp")
    synth_o = os.path.join(BUILD, "synth.o")
    objs.append(synth_o)
    if force or _stale(synth_o, [synth_src, os.path.join(ROOT, "synth", "synth.h")]):
        jobs.append(["g++", "-O2", "-std=c++17", "-fPIC", "-pthread", "-c", synth_src, "-o", synth_o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stdout + r.stderr

    logs = []
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
            logs = list(ex.map(run, jobs))
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        run([cc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lpthread"])
        os.replace(tmp, LIB)
    if verbose:
        print("\n".join(logs))
    return LIB


if __name__ == "__main__":
    import sys
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
