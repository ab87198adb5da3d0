"""Compile the C oracles (test infrastructure): the forward into
oracle/libfa2_oracle.so and its gradient into oracle/libfa2_bwd_oracle.so.

Plain gcc, -O2, no fast-math and no host-specific flags, so the same source
gives the same results on x86-64 and AArch64 hosts.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fa2_oracle.c")
LIB = os.path.join(HERE, "libfa2_oracle.so")
BWD_SRC = os.path.join(HERE, "fa2_bwd_oracle.c")
BWD_LIB = os.path.join(HERE, "libfa2_bwd_oracle.so")


def compile_c(src: str, lib: str) -> None:
    tmp = lib + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11", "-fPIC",
           "-shared", "-pthread", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)


def _stale(src: str, lib: str) -> bool:
    return not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src)


def build(force: bool = False) -> str:
    """Build both oracle libraries if needed; returns the forward library's path."""
    for src, lib in ((SRC, LIB), (BWD_SRC, BWD_LIB)):
        if force or _stale(src, lib):
            compile_c(src, lib)
    return LIB


def build_bwd(force: bool = False) -> str:
    build(force)
    return BWD_LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv)
    print(LIB)
    print(BWD_LIB)
