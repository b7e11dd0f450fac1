"""Build libmqa.so (the CUDA library behind the C ABI in include/mqa.h).

Compiles every translation unit under ``csrc/`` for sm_103a with nvcc, in
parallel, and links them into ``fp8_mqa_indexer_gb300/libmqa.so``.  Runs on a
machine without a GPU (nvcc cross-compiles); the CUDA runtime is linked
statically and the driver entry point is fetched at run time, so the library
loads on hosts that have no CUDA driver.

    python -m fp8_mqa_indexer_gb300.build [--force]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmqa.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
UNITS = ["mqa_api.cu", "mqa_dense.cu", "mqa_dense_bf16.cu", "mqa_dense_cand.cu", "mqa_dense_mx.cu",
         "mqa_paged.cu", "mqa_paged_bf16.cu", "mqa_paged_mx.cu", "mqa_topk.cu"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmqa.so")


def _sources_mtime() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _sources_mtime():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE]
    if verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(unit: str) -> str:
        obj = os.path.join(BUILD, unit.replace(".cu", ".o"))
        cmd = [cc] + flags + ["-c", os.path.join(CSRC, unit), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {unit}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(len(UNITS)) as ex:
        objs = list(ex.map(compile_one, UNITS))
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([cc, "-shared"] + ARCH + ["-o", tmp] + objs, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose))
