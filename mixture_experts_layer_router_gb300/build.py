"""Build liblatentmoe.so in-tree with nvcc for sm_103a.

The translation units are compiled in parallel, then linked into
``mixture_experts_layer_router_gb300/_build/liblatentmoe.so`` with the CUDA
runtime linked statically. A unit is rebuilt when it or any header is newer
than its object file.

``build(variant="bounds")`` builds the bounds-checked debug library
``_build/bounds/liblatentmoe.so`` (compiled with -DLMOE_BOUNDS): every
epilogue store, scatter write and combine read checks its row against its
buffer, skips an access outside it and sets LATENTMOE_STATUS_BOUNDS. It is
the stand-in for a memory checker; the regular library is unchanged by it.
"""
from __future__ import annotations

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
LIB = os.path.join(BUILD, "liblatentmoe.so")

SOURCES = ["api.cu", "route.cu", "combine.cu", "gemm_bf16.cu", "gemm_f32.cu",
           "gemm_swiglu.cu", "gemm_scatter.cu", "gemm_scatter8.cu", "gemm_grouped.cu", "gemm_grouped2.cu", "gemm_fused.cu",
           "pack.cu",
           "router.cu", "route_static.cu", "fp8.cu", "multiround.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblatentmoe")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


VARIANTS = {None: [], "bounds": ["-DLMOE_BOUNDS"]}


def lib_path(variant=None) -> str:
    return LIB if variant is None else os.path.join(BUILD, variant, "liblatentmoe.so")


def _compile(nvcc: str, src: str, extra, out_dir: str = BUILD) -> str:
    obj = os.path.join(out_dir, os.path.basename(src) + ".o")
    if _stale(obj, [src] + _headers()):
        cmd = [nvcc, *FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if r.stderr.strip() and os.environ.get("LATENTMOE_BUILD_VERBOSE"):
            sys.stderr.write(r.stderr)
    return obj


def build(verbose: bool = False, extra_flags=(), variant=None) -> str:
    """Compile every unit and link the shared library; returns its path.
    variant: None (the library) or "bounds" (the bounds-checked debug build,
    kept in its own folder)."""
    out_dir = BUILD if variant is None else os.path.join(BUILD, variant)
    lib = lib_path(variant)
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    flags = list(VARIANTS[variant]) + list(extra_flags)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    workers = min(len(srcs), max(1, os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, flags, out_dir), srcs))
    if _stale(lib, objs):
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", lib, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    if verbose:
        print(f"built {lib}")
    return lib


if __name__ == "__main__":
    build(verbose=True, variant=sys.argv[1] if len(sys.argv) > 1 else None)
