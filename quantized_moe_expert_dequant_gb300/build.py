"""Builds libmoe_decode.so in-tree with nvcc for sm_103a only.

    python -m quantized_moe_expert_dequant_gb300.build

Each translation unit compiles in parallel into _build/, then one nvcc link writes
quantized_moe_expert_dequant_gb300/libmoe_decode.so.  The CUDA runtime is linked dynamically so
that a process which already loaded PyTorch shares one runtime with it.
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
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmoe_decode.so")
# The timeline build: the same sources with MOE_TIMELINE defined, so that the column-split kernel
# records per-CTA, per-layer time stamps (moe_timeline.cuh) readable through moe_stack_timeline.
LIB_TIMELINE = os.path.join(PKG, "libmoe_decode_timeline.so")
SOURCES = ["moe_kernels_g4.cu", "moe_kernels_g6.cu", "moe_kernels_g8.cu", "moe_grouped_g4.cu",
           "moe_grouped_g6.cu", "moe_grouped_g8.cu", "moe_cols_g4.cu", "moe_cols_g6.cu",
           "moe_cols_g8.cu", "moe_kernels.cu", "moe_mma.cu",
           "moe_api.cu", "moe_pack.cpp", "synth.cu", "gemv.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe_decode.so")
    return path


def cuda_lib_dir() -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc()))), "lib64")


def _compile(src: str, verbose: bool, timeline: bool = False) -> str:
    out_dir = os.path.join(BUILD, "timeline") if timeline else BUILD
    obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj, "-O3", "-lineinfo", "-std=c++17",
           "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC] + ARCH
    if timeline:
        cmd.append("-DMOE_TIMELINE")
    if verbose:
        cmd.append("-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
        os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)] + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, timeline: bool = False) -> str:
    lib = LIB_TIMELINE if timeline else LIB
    if not force and not _stale(lib):
        return lib
    os.makedirs(os.path.join(BUILD, "timeline") if timeline else BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, timeline), SOURCES))
    tmp = lib + f".{os.getpid()}.tmp"
    cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + [
        "-cudart", "shared", "-Xlinker", "-rpath=" + cuda_lib_dir()]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                timeline="--timeline" in sys.argv))
