"""Build of the CUDA library (sm_103a) in-tree: one nvcc job per source, then a shared link."""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libmoe_resident.so")
OBJ_DIR = os.path.join(PKG, "_build")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
                 "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _needs(out: str, deps: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, obj: str, extra: list[str]) -> None:
    tmp = obj + f".tmp{os.getpid()}"
    subprocess.check_call([NVCC] + CFLAGS + extra + ["-c", src, "-o", tmp])
    os.replace(tmp, obj)


def build_library(sources: list[str], lib: str, obj_dir: str, headers: list[str], extra: list[str] = (),
                  jobs: int = 8, verbose_ptxas: bool = False) -> str:
    os.makedirs(obj_dir, exist_ok=True)
    extra = list(extra) + (["-Xptxas", "-v"] if verbose_ptxas else [])
    objs = []
    todo = []
    for src in sources:
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        objs.append(obj)
        if verbose_ptxas or _needs(obj, [src] + headers):
            todo.append((src, obj))
    if todo:
        with cf.ThreadPoolExecutor(max_workers=min(jobs, len(todo))) as ex:
            for f in [ex.submit(_compile, s, o, extra) for s, o in todo]:
                f.result()
    if todo or _needs(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.check_call([NVCC] + ARCH + ["-shared", "-o", tmp] + objs + ["-ldl", "-lpthread", "-lrt"])
        os.replace(tmp, lib)
    return lib


MICROBENCH_SRC = os.path.join(PKG, "microbench", "mma_scale_rate.cu")
MICROBENCH_BIN = os.path.join(PKG, "microbench", "mma_scale_rate")


def build_microbench() -> str:
    """The tensor-pipe microbenchmark that bench.py runs for the measured FP4 MMA rate."""
    if _needs(MICROBENCH_BIN, [MICROBENCH_SRC, os.path.join(CSRC, "common.cuh")]):
        tmp = MICROBENCH_BIN + f".tmp{os.getpid()}"
        subprocess.check_call([NVCC] + ARCH + ["-O3", "-std=c++17", "-I", os.path.join(ROOT, "include"), "-o", tmp,
                               MICROBENCH_SRC])
        os.replace(tmp, MICROBENCH_BIN)
    return MICROBENCH_BIN


def build(verbose_ptxas: bool = False) -> str:
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [os.path.join(ROOT, "include", "moe_resident.h")]
    return build_library(sources, LIB, OBJ_DIR, headers, verbose_ptxas=verbose_ptxas)


if __name__ == "__main__":
    import sys
    print(build(verbose_ptxas="-v" in sys.argv))
