"""Build libpagedkv.so in-tree with nvcc for sm_103a (no CMake, no torch
extension machinery): each .cu file compiles in parallel, then one shared
link against the static CUDA runtime.

    python -m paged_kv_cache_104_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpagedkv.so")
SOURCES = ["abi.cu", "append.cu", "decode.cu", "decode_fp8.cu", "decode_mla.cu", "decode_mma.cu",
           "gemm_heads.cu", "decode_noalloc.cu", "host_cache.cu", "l2_flush.cu", "prefill_pair.cu",
           "prefix_cache.cpp", "tmap.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hdrs + [os.path.join(INCLUDE, "pagedkv.h")]


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    dep_time = max(os.path.getmtime(p) for p in _deps())
    procs, objs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        objs.append(o)
        if not force and os.path.exists(o) and os.path.getmtime(o) >= max(os.path.getmtime(s), dep_time):
            continue
        cmd = [nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
               "-I", INCLUDE, "-I", CSRC, "-c", s, "-o", o]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((src, text))
        elif verbose and text:
            print(f"--- {src}\n{text}", file=sys.stderr)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(f"--- {s}\n{t}" for s, t in failed))
    if force or procs or not os.path.exists(LIB):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"], check=True)
        os.replace(tmp, LIB)
    return LIB


# A test-only build of the library: the same objects but decode_mma.cu
# compiled with PKV_TEST_WAIT_TIMEOUT, which shortens every wait limit of that
# file to about 2 ms and makes the decode kernel's producer withhold its
# copies, so a test can see a wait run out and the kernel return with
# PKV_DEVERR_TIMEOUT.  Never loaded by the product.
WAIT_TEST_DIR = os.path.join(BUILD, "wait_test")
WAIT_TEST_LIB = os.path.join(WAIT_TEST_DIR, "libpagedkv_wait_test.so")


def build_wait_test() -> str:
    build()
    os.makedirs(WAIT_TEST_DIR, exist_ok=True)
    src = os.path.join(CSRC, "decode_mma.cu")
    obj = os.path.join(WAIT_TEST_DIR, "decode_mma.o")
    dep_time = max([os.path.getmtime(p) for p in _deps()] + [os.path.getmtime(src)])
    if not os.path.exists(obj) or os.path.getmtime(obj) < dep_time:
        subprocess.run([nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
                        "-DPKV_TEST_WAIT_TIMEOUT", "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj],
                       check=True)
    objs = [obj] + [os.path.join(BUILD, os.path.splitext(f)[0] + ".o") for f in SOURCES
                    if f != "decode_mma.cu"]
    if not os.path.exists(WAIT_TEST_LIB) or os.path.getmtime(WAIT_TEST_LIB) < max(
            os.path.getmtime(o) for o in objs):
        tmp = WAIT_TEST_LIB + f".tmp{os.getpid()}"
        subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"], check=True)
        os.replace(tmp, WAIT_TEST_LIB)
    return WAIT_TEST_LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    args = ap.parse_args()
    print(build(args.force, args.verbose))
