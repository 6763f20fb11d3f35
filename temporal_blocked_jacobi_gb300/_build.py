"""Build the solver's C-ABI shared library for sm_103a with nvcc.

The library is built in-tree (temporal_blocked_jacobi_gb300/libtbjacobi.so);
objects go to temporal_blocked_jacobi_gb300/_build/. Translation units are
compiled in parallel. The CUDA runtime is linked statically and the driver
entry point for TMA descriptors is looked up at run time, so the library has
no link-time dependency on libcuda.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtbjacobi.so")
# The bounds-checked variant (JACOBI_BOUNDS_CHECK; see include/jacobi.h):
# same sources, its own objects.
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libtbjacobi_checked.so")
# The four kernels_etb_part*.cu units come first: they take longest.
SOURCES = ["kernels_etb_part0.cu", "kernels_etb_part1.cu", "kernels_etb_part2.cu",
           "kernels_etb_part3.cu", "kernels_etb.cu", "kernels_etbs.cu",
           "kernels_sync.cu",
           "kernels_tiled.cu", "kernels_ba.cu", "kernels_bar.cu", "fastdiv.cu",
           "jacobi_abi.cu", "residual_noalloc.cu", "adapt.cu"]
HEADERS = [os.path.join(CSRC, "jacobi_kernels.cuh"),
           os.path.join(CSRC, "etb_kernels.cuh"),
           os.path.join(ROOT, "include", "jacobi.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    "-O3", "-std=c++17", *ARCH, "-lineinfo",
    # IEEE arithmetic everywhere: no multiply-add contraction, subnormals
    # kept, correctly rounded division.
    "-fmad=false", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
    "-Xcompiler", "-fPIC,-ffp-contract=off",
    "-Xptxas", "-warn-spills",
    "-I", os.path.join(ROOT, "include"),
]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build")
    return path


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [__file__]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile and link libtbjacobi.so (checked: libtbjacobi_checked.so) if
    any source changed. Returns its path."""
    lib, build_dir = (LIB_CHECKED, BUILD_CHECKED) if checked else (LIB, BUILD)
    if not force and not _stale(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + (["-DJACOBI_BOUNDS_CHECK"] if checked else [])

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            print(res.stdout + res.stderr, flush=True)
        return obj

    workers = max(1, min(len(SOURCES), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}{res.stderr}")
    os.replace(tmp, lib)
    return lib


def build_all(force: bool = False, verbose: bool = False):
    """Both libraries, compiled side by side. Returns their paths."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        futs = [ex.submit(build, force, verbose, c) for c in (False, True)]
        return [f.result() for f in futs]


if __name__ == "__main__":
    print(build_all(force=True, verbose=True))
