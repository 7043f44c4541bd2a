"""Build liblinattn.so in-tree with nvcc for sm_103a (GB300).

Each .cu translation unit in csrc/ is compiled to an object file in
_build/ (in parallel), then linked into recurrent_lm_gb300/liblinattn.so.
The CUDA runtime is linked statically; the driver API (tensor-map encoding)
is reached through cudaGetDriverEntryPoint, so no -lcuda is needed.

Usage:  python -m recurrent_lm_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "liblinattn.so")
TRACE_LIB = os.path.join(PKG, "liblinattn_trace.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblinattn.so")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.h")) +
            glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date(lib: str = None) -> bool:
    lib = lib or LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _compile(src: str, verbose: bool, extra, build_dir: str = BUILD_DIR) -> str:
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)
    return obj


def build(force: bool = False, verbose: bool = False, extra=(), trace: bool = False) -> str:
    """Compile every csrc/*.cu for sm_103a and link liblinattn.so; returns its path.

    trace=True builds liblinattn_trace.so instead, with the per-role timeline
    of the tensor-core prefill compiled in (-DLA_TRACE)."""
    lib = TRACE_LIB if trace else LIB
    build_dir = os.path.join(BUILD_DIR, "trace") if trace else BUILD_DIR
    extra = list(extra) + (["-DLA_TRACE"] if trace else [])
    if not force and up_to_date(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, extra, build_dir), srcs))
    tmp = lib + f".tmp{os.getpid()}"
    # cuBLASLt (the d' = 24, 32 tensor-core path), found next to the toolkit's nvcc
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(nvcc())), "lib64")
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcublasLt", "-Xlinker", "-rpath", "-Xlinker", cuda_lib]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-v", action="store_true", help="print register / spill usage")
    ap.add_argument("--trace", action="store_true", help="build liblinattn_trace.so")
    a = ap.parse_args()
    extra = ["-Xptxas", "-v"] if a.ptxas_v else []
    print(build(force=a.force or a.ptxas_v, verbose=a.verbose or a.ptxas_v, extra=extra,
                trace=a.trace))
    sys.exit(0)
