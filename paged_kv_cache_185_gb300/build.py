"""Build libwllm.so (the sm_103a CUDA library behind include/wllm.h) in-tree.

    python -m paged_kv_cache_185_gb300.build [--force] [--verbose]

Each translation unit is compiled by nvcc in parallel into ``_build/`` and
linked into ``paged_kv_cache_185_gb300/libwllm.so`` against the shared CUDA
runtime.  Only ``sm_103a`` code is generated.  A rebuild happens when any source
or header is newer than the library.
"""
from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libwllm.so")

SOURCES = ["api.cu", "append.cu", "decode_bf16.cu", "decode_f16.cu", "decode_f32.cu", "decode_f8_f16.cu",
           "decode_f8_bf16.cu", "prefill.cu", "prefill_tc.cu", "block_manager.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    files += glob.glob(os.path.join(CSRC, "*.inc")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    common = [nvcc, *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-I", INCLUDE, "-I", CSRC]
    if ptxas_verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src: str):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [*common, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    failed = False
    for src, _, r in results:
        if verbose or ptxas_verbose or r.returncode != 0:
            sys.stderr.write(f"--- {src}\n{r.stdout}{r.stderr}")
        failed |= r.returncode != 0
    if failed:
        raise RuntimeError("nvcc failed")
    tmp = LIB + f".{os.getpid()}.tmp"
    link = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *[o for _, o, _ in results],
            "-Xlinker", "-rpath," + _cuda_lib_dir(nvcc), "-Xlinker", "-z,defs"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("link failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, ptxas_verbose=a.ptxas_verbose))
