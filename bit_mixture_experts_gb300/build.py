"""Build libmoe_w4.so in-tree with nvcc for sm_103a.

Each .cu under csrc/ is compiled to an object in parallel, then linked into
bit_mixture_experts_gb300/libmoe_w4.so (CUDA runtime linked statically).
Objects go to bit_mixture_experts_gb300/_build/.  Rebuilds only what changed.
With --trace the same sources are built with -DMOE_TRACE into
libmoe_w4_trace.so (objects in _build_trace/): the tensor-core kernels then
record their wait statistics (moe_trace_read; `python -m
bit_mixture_experts_gb300.trace` reports them).

    python -m bit_mixture_experts_gb300.build [--force] [--verbose] [--trace]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe_w4.so")
BUILD_TRACE = os.path.join(PKG, "_build_trace")
LIB_TRACE = os.path.join(PKG, "libmoe_w4_trace.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
                     "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe_w4.so")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, force: bool, verbose: bool, extra=(), build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    if force or _stale(obj, [src, *_headers(), __file__]):
        cmd = [nvcc(), *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
    return obj


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, trace: bool = False) -> str:
    build_dir, lib = (BUILD_TRACE, LIB_TRACE) if trace else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    srcs = _sources()
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DMOE_TRACE"] if trace else [])
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, force or ptxas_info, verbose or ptxas_info, extra, build_dir), srcs))
    if force or _stale(lib, objs):
        tmp = lib + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print -Xptxas -v register/smem usage")
    ap.add_argument("--trace", action="store_true", help="build libmoe_w4_trace.so (-DMOE_TRACE) instead")
    a = ap.parse_args(argv)
    print(build(a.force, a.verbose, a.ptxas_info, a.trace))


if __name__ == "__main__":
    sys.exit(main())
