"""Builds libtopk.so in-tree for sm_103a (nvcc; no cmake, no torch extension).

Each translation unit compiles in its own process, in parallel, then nvcc
links the shared library next to this file. Run ``python -m
sparse_attention_row_gb300.build`` or call ``build_library()``.
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
LIB = os.path.join(HERE, "libtopk.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["topk_kernel.cu", "topk_kernel_pair.cu", "topk_kernel_small.cu", "topk_short.cu", "topk_short16.cu", "topk_sort.cu",
           "topk_api.cu",
           "topk_static.cu", "planner.cpp"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libtopk")
    return cand


def _compile(src: str, verbose_ptxas: bool) -> str:
    nvcc = _nvcc()
    path = os.path.join(CSRC, src)
    obj = os.path.join(OUT_DIR, src + ".o")
    cmd = [nvcc, "-c", path, "-o", obj, "-std=c++17", "-O3", "-Xcompiler", "-fPIC,-O2",
           "-I", os.path.join(HERE, "..", "include")]
    if src.endswith(".cu"):
        cmd += ARCH + ["-lineinfo"]
        if verbose_ptxas:
            cmd += ["-Xptxas", "-v"]
    else:
        cmd = [nvcc, "-x", "c++", "-c", path, "-o", obj, "-std=c++17", "-O2", "-Xcompiler", "-fPIC",
               "-I", os.path.join(HERE, "..", "include")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"compiling {src} failed:\n{res.stdout}\n{res.stderr}")
    if verbose_ptxas and res.stderr:
        sys.stderr.write(res.stderr)
    return obj


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(HERE, "..", "include", "libtopk.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build_library(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compiles libtopk.so if any source is newer than it; returns its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas), SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [_nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-lcudart_static", "-lrt", "-ldl", "-lpthread"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"linking libtopk.so failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
