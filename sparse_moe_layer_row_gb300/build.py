"""Build libmoeblock.so (CUDA, sm_103a) in-tree, under sparse_moe_layer_row_gb300/_build/.

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library with the C ABI of include/moe_block.h.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libmoeblock.so")
SOURCES = ["api.cu", "router.cu", "router_tc.cu", "coreset.cu", "scatter.cu",
           "gemm.cu", "gemm_pair.cu", "noalloc.cu"]
HEADERS = ["common.cuh", "kernels.cuh", "route_common.cuh", "coreset_dev.cuh", "scatter_dev.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    root = os.path.dirname(HERE)
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS] +
            [os.path.join(root, "include", "moe_block.h"), os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    cc = nvcc()
    objs = []
    logs = {}

    def compile_one(src):
        obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for src, obj, r in ex.map(compile_one, SOURCES):
            logs[src] = r.stdout + r.stderr
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{logs[src]}")
            objs.append(obj)
    with open(os.path.join(OUT_DIR, "ptxas.log"), "w") as f:
        for src in SOURCES:
            f.write(f"==== {src}\n{logs[src]}\n")
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([cc, *ARCH, "-shared", *objs, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        print(open(os.path.join(OUT_DIR, "ptxas.log")).read())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
