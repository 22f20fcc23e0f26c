"""Ahead-of-time build of libdg.so (sm_103a) next to this file.

Each CUDA translation unit is compiled in parallel with nvcc and the objects are linked into
one shared library with a plain C ABI (include/dg.h).  The CUDA runtime is linked
statically; the driver's tensor-map encoder is reached through the runtime's driver entry
point, so no libcuda link is needed at build time.  `build(debug=True)` makes the debug build
libdg_debug.so (-DDG_DEBUG=1: kernels check their computed indices, see dg_debug_word), which
the binding loads instead when the environment sets DG_DEBUG=1.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdg.so")
DEBUG_BUILD_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB = os.path.join(PKG, "libdg_debug.so")
SOURCES = ["host_common.cu", "quant.cu", "gemm.cu", "gemm_mx.cu", "gemm_bf16.cu", "kgrouped.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "dg.h"))
    files.append(os.path.abspath(__file__))
    return files


def library_path(debug: bool = False) -> str:
    return DEBUG_LIB if debug else LIB


def is_stale(debug: bool = False) -> bool:
    lib = library_path(debug)
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _remove_orphan_objects(build_dir: str) -> None:
    """Delete objects in the build folder whose source is no longer compiled, so that nothing
    stale lies beside the library."""
    keep = {os.path.splitext(s)[0] + ".o" for s in SOURCES}
    for f in os.listdir(build_dir):
        if f.endswith(".o") and f not in keep:
            os.remove(os.path.join(build_dir, f))


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile csrc/*.cu for sm_103a and link libdg.so (libdg_debug.so if `debug`); returns its
    path."""
    lib = library_path(debug)
    if not force and not is_stale(debug):
        return lib
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    os.makedirs(build_dir, exist_ok=True)
    _remove_orphan_objects(build_dir)
    nvcc = _nvcc()
    flags = NVCC_FLAGS + (["-DDG_DEBUG=1"] if debug else [])

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
