"""In-tree build of the CUDA library libmoe_b300.so (sm_103a) with nvcc.

    python -m sparsely_gated_mixture_top_b300.build [--ptxas-verbose]

Each .cu file under csrc/ is compiled to an object in csrc/_build/ (in
parallel), then linked into sparsely_gated_mixture_top_b300/libmoe_b300.so.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "libmoe_b300.so")
BUILD = os.path.join(CSRC, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
                  glob.glob(os.path.join(ROOT, "include", "*.h")))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    hdrs = _headers()
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in srcs]
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []

    def compile_one(src, obj):
        if force or verbose_ptxas or _stale(obj, [src] + hdrs):
            cmd = ["nvcc", *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
            return r.stderr
        return ""

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        logs = list(ex.map(compile_one, srcs, objs))
    if verbose_ptxas:
        for src, log in zip(srcs, logs):
            sys.stderr.write(f"== {os.path.basename(src)}\n{log}")
    if force or _stale(OUT, objs):
        cmd = ["nvcc", *ARCH, "-shared", "-o", OUT, *objs]
        subprocess.check_call(cmd)
    return OUT


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="--ptxas-verbose" in sys.argv)
    print(OUT)
