"""Builds libfa_gb300.so in-tree with nvcc for sm_103a (no torch extension
machinery: the library is a plain C-ABI shared object)."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB_PATH = os.path.join(HERE, "libfa_gb300.so")
SOURCES = ["fa_api.cu"]
DEPENDS = ["fa_api.cu", "fa_fwd_kernel.cuh", "fa_bwd_kernel.cuh", "fa_fp8_quant.cuh", "ptx_sm103.cuh", os.path.join("..", "..", "include", "fa.h")]


def nvcc_command(out: str = LIB_PATH, extra=()):
    return ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
            "-shared", "-Xcompiler", "-fPIC", "-cudart", "static", *extra,
            "-o", out, *[os.path.join(CSRC, s) for s in SOURCES]]


def up_to_date(out: str = LIB_PATH) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(os.path.join(CSRC, d)) <= t for d in DEPENDS)


def build(force: bool = False, out: str = LIB_PATH, verbose: bool = False) -> str:
    if force or not up_to_date(out):
        extra = ("-Xptxas", "-v") if verbose else ()
        subprocess.run(nvcc_command(out, extra), check=True)
    return out


if __name__ == "__main__":
    build(force=True, verbose=True)
