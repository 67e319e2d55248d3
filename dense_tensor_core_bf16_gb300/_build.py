"""Compile the CUDA library in-tree: csrc/*.cu, csrc/*.cpp -> _build/libgemm_bf16.so.

One nvcc invocation for sm_103a (``-gencode arch=compute_103a,code=sm_103a``),
host code position-independent, the CUDA runtime linked statically and the
driver API reached at run time through cudaGetDriverEntryPointByVersion, so
the library loads on a machine without a GPU.
"""
from __future__ import annotations

import os
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libgemm_bf16.so")

SOURCES = ["gemm_bf16.cu", "plan.cpp", "host_pipeline.cpp"]
NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
]


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return files


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build_library(force: bool = False, verbose: bool = False) -> str:
    if not force and not is_stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc, *NVCC_FLAGS, "-I", INCLUDE, "-o", tmp] + [os.path.join(CSRC, s) for s in SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.check_call(cmd)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH
