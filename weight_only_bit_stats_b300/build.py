"""Build libawq_b300.so in-tree for sm_103a (B300) with nvcc.

Each CUDA source is compiled to an object in ``_build/`` (in parallel,
skipped when up to date), then linked into ``_build/libawq_b300.so`` with
the CUDA runtime linked statically, so the library loads on a machine without
a GPU (calls then fail with AWQ_ERR_DEVICE / AWQ_ERR_CUDA).

Usage: ``python -m weight_only_bit_stats_b300.build [-v]`` (``-v`` prints the
ptxas register / spill report).
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libawq_b300.so")
SOURCES = ["capi.cu", "stats.cu", "quant.cu", "gemv.cu", "gemv_tiles.cu", "gemv3.cu", "tc.cu",
           "gram.cu", "search_noalloc.cu"]
HEADERS = ["common.cuh", "kernels.cuh", "int3.cuh", "decode.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest_dep() -> float:
    deps = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "awq.h")]
    return max(os.path.getmtime(p) for p in deps)


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(BUILD, src.replace(".cu", ".o"))
    path = os.path.join(CSRC, src)
    if (not verbose and os.path.exists(obj)
            and os.path.getmtime(obj) >= max(os.path.getmtime(path), _newest_dep())):
        return obj
    cmd = [_nvcc(), *ARCH, *FLAGS, "-c", path, "-o", obj + ".tmp"]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    if verbose and res.stderr:
        sys.stderr.write(res.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(verbose: bool = False) -> str:
    """Compile and link the library if any source changed; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    if (not os.path.exists(LIB) or
            os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs)):
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = [_nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-cudart", "static",
               *objs, "-o", tmp]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
