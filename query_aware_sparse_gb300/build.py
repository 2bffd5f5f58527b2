"""Builds libquest.so in-tree with nvcc for sm_103a (GB300).

Each .cu file compiles to an object in parallel, then one shared library is
linked (static CUDA runtime). Objects are rebuilt only when a source or header
is newer. Usable as ``python -m query_aware_sparse_gb300.build``.
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
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libquest.so")
SOURCES = ["quest_api.cu", "append.cu", "score.cu", "select.cu", "attn.cu", "step.cu",
           "step_f32_d64.cu", "step_f32_d128.cu", "step_f16_d64.cu", "step_f16_d128.cu",
           "step_e4m3_d64.cu", "step_e4m3_d128.cu", "noalloc.cu", "diag.cu", "union.cu",
           "cstep_f32_d64.cu", "cstep_f32_d128.cu", "cstep_f16_d64.cu", "cstep_f16_d128.cu",
           "cstep_e4m3_d64.cu", "cstep_e4m3_d128.cu"]
HEADERS = [os.path.join(CSRC, h) for h in ("common.cuh", "internal.h", "topk.cuh", "attn_dev.cuh",
                                           "attn_mma.cuh", "step_impl.cuh",
                                           "cstep_impl.cuh")] + [
           os.path.join(ROOT, "include", "quest.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
                "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libquest needs the CUDA toolkit to build")


def _mtime(p):
    return os.path.getmtime(p) if os.path.exists(p) else 0.0


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile and link libquest.so; returns its path."""
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    hdr_time = max(_mtime(h) for h in HEADERS)
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _mtime(o) < max(_mtime(s), hdr_time):
            jobs.append([nvcc, *FLAGS, *extra_flags, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {cmd[-3]}")
        return r

    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            list(ex.map(run, jobs))
    if force or jobs or _mtime(LIB) < max(_mtime(o) for o in objs):
        tmp = LIB + ".tmp"
        run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
