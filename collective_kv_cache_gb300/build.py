"""Build the C-ABI library libtd.so in-tree for sm_103a (GB300).

Each CUDA translation unit is compiled by nvcc in parallel, the host layer by g++, and the
objects are linked into collective_kv_cache_gb300/libtd.so (static CUDA runtime).
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
INC = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "libtd.so")
BUILD_DIR = os.path.join(ROOT, "_build")

CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CU_FLAGS = ["-O3", "-lineinfo", "--fmad=false", "-std=c++17", "-Xcompiler", "-fPIC",
            "-Xcompiler", "-ffp-contract=off", "-Xptxas", "-v"]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-ffp-contract=off", "-fno-fast-math", "-Wall",
             "-Wextra"]

CU_SOURCES = ["k_rerotate.cu", "k_select.cu", "k_master.cu", "k_encode.cu", "k_restore.cu",
              "k_variants.cu", "td_noalloc.cu", "k_attention.cu"]
CXX_SOURCES = ["td_host.cpp", "td_rounds.cpp"]
HEADERS = ["td_internal.h", "td_device.cuh"]


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in CU_SOURCES + CXX_SOURCES + HEADERS]
    paths.append(os.path.join(INC, "td.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def _run(cmd, log):
    p = subprocess.run(cmd, capture_output=True, text=True)
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + p.stdout + p.stderr)
    if p.returncode != 0:
        sys.stderr.write(p.stdout + p.stderr)
        raise RuntimeError(f"build step failed: {' '.join(cmd)}")
    return log


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(OUT) and os.path.getmtime(OUT) >= _newest_input():
        return OUT
    if not os.path.exists(NVCC):
        raise RuntimeError(f"nvcc not found at {NVCC}")
    os.makedirs(BUILD_DIR, exist_ok=True)
    inc = ["-I", INC, "-I", CSRC]
    jobs = []
    objs = []
    for src in CU_SOURCES:
        obj = os.path.join(BUILD_DIR, src + ".o")
        objs.append(obj)
        jobs.append(([NVCC, *ARCH, *CU_FLAGS, *inc, "-c", os.path.join(CSRC, src), "-o", obj],
                     obj + ".log"))
    cxx = shutil.which("g++") or "g++"
    for src in CXX_SOURCES:
        obj = os.path.join(BUILD_DIR, src + ".o")
        objs.append(obj)
        jobs.append(([cxx, *CXX_FLAGS, *inc, "-I", os.path.join(CUDA_HOME, "include"), "-c",
                      os.path.join(CSRC, src), "-o", obj], obj + ".log"))
    with cf.ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
        logs = list(ex.map(lambda j: _run(*j), jobs))
    tmp = OUT + ".tmp"
    _run([NVCC, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-lrt", "-ldl",
          "-lpthread"], os.path.join(BUILD_DIR, "link.log"))
    os.replace(tmp, OUT)
    if verbose:
        for lg in logs:
            with open(lg) as f:
                sys.stdout.write(f.read())
    return OUT


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
