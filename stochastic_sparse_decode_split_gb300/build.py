"""Builds libsanta.so in-tree for sm_103a with nvcc (no GPU needed).

    python -m stochastic_sparse_decode_split_gb300.build [--force]

Translation units compile in parallel, then link into
``stochastic_sparse_decode_split_gb300/_build/libsanta.so`` against the shared
CUDA runtime (the same libcudart.so.13 PyTorch loads).
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libsanta.so")
SOURCES = ["santa_api.cu", "santa_score.cu", "santa_sample.cu", "santa_fused.cu", "santa_fused_bf16.cu", "santa_fused_fp16.cu",
           "santa_flash.cu", "santa_static.cu", "santa_tiled.cu", "santa_bernoulli.cu", "santa_probe.cu"]
HEADERS = ["santa_common.cuh", "santa_flash.cuh", "santa_fused.cuh", "santa_grid.cuh", "santa_launch.h", "santa_part.cuh",
           "santa_seq.cuh", "santa_stream.cuh", "santa_tma.cuh", "santa_window.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; set NVCC or add the CUDA toolkit to PATH")
    return cand


def _cuda_lib_dir(nv: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nv))), "lib64")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    nv = nvcc()
    common_deps = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "santa.h"),
                                                              os.path.abspath(__file__)]
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
                    "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")] + list(extra_flags or [])
    if os.environ.get("SANTA_PTXAS_VERBOSE"):
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        srcp = os.path.join(CSRC, src)
        if force or _stale(obj, [srcp] + common_deps):
            cmd = [nv] + flags + ["-c", srcp, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
            if verbose or os.environ.get("SANTA_PTXAS_VERBOSE"):
                sys.stderr.write(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nv] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs + [
            "-Xlinker", "-rpath," + _cuda_lib_dir(nv)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
