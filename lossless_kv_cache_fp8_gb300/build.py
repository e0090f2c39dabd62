"""Builds libskv.so in-tree with nvcc for sm_103a (no torch extension machinery)."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "skv.cu")
HDR = os.path.join(ROOT, "include", "skv.h")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libskv.so")
LIB_CHECKED = os.path.join(OUT_DIR, "libskv_checked.so")   # -DSKV_CHECKED=1: bounds-checked kernels
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """libskv.so (or, checked=True, libskv_checked.so with the bounds checks)"""
    os.makedirs(OUT_DIR, exist_ok=True)
    out = LIB_CHECKED if checked else LIB
    newest = max(os.path.getmtime(SRC), os.path.getmtime(HDR))
    if not force and os.path.exists(out) and os.path.getmtime(out) >= newest:
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "--shared", "-Xcompiler", "-fPIC",
           "-cudart", "static", "-I", os.path.join(ROOT, "include"), "-o", tmp, SRC]
    if checked:
        cmd.insert(1, "-DSKV_CHECKED=1")
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.check_call(cmd)
    os.replace(tmp, out)
    return out
