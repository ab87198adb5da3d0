"""Build the sm_103a forward library in-tree: attention_forward_03_gb300/libfa2_gb300.so.

Each CUDA translation unit is compiled in parallel with nvcc for sm_103a only,
then linked into one shared library (CUDA runtime linked statically). No cmake,
no torch extension machinery: the product is a plain C-ABI shared object.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libfa2_gb300.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
SOURCES = ["fa2_api.cu", "fa2_noalloc.cu", "fa2_host.cu", "fa2_fwd_d32.cu", "fa2_fwd_d64.cu", "fa2_fwd_d96.cu",
           "fa2_fwd_d128.cu", "fa2_fwd_d256.cu",
           "fa2_fwd_d512.cu", "fa2_fwd_d1024.cu", "fa2_bwd_api.cu",
           "fa2_bwd_d32.cu", "fa2_bwd_d64.cu", "fa2_bwd_d96.cu", "fa2_bwd_d128.cu"]
GENCODE = "arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")
    return path


def _flags(verbose_ptxas: bool) -> list[str]:
    # hidden visibility: only the C ABI (FA2_API in fa2.h) is exported, so two
    # copies of the library in one process never share a symbol
    f = ["-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
         "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _inputs_newer(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "fa2.h"))
    objs = []
    todo = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _inputs_newer(o, [s] + headers):
            todo.append((s, o))

    def compile_one(so):
        s, o = so
        cmd = [nvcc(), *_flags(verbose_ptxas), "-c", s, "-o", o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(s)}:\n{r.stdout}\n{r.stderr}")
        return r.stdout + r.stderr

    logs = []
    if todo:
        with cf.ThreadPoolExecutor(max_workers=jobs or len(todo)) as ex:
            logs = list(ex.map(compile_one, todo))
    if todo or force or not os.path.exists(LIB_PATH):
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [nvcc(), "-gencode", GENCODE, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB_PATH)
    if verbose_ptxas:
        for log in logs:
            sys.stdout.write(log)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
