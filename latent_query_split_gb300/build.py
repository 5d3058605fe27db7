"""Builds the C-ABI CUDA library libflare.so in-tree (sm_103a, nvcc only).

Each translation unit under csrc/ compiles in parallel; the objects link into
latent_query_split_gb300/_build/libflare.so. Rebuilds only when a source or
header is newer than the library.

build(debug=True) makes the checking variant _build_debug/libflare.so
(-DFLARE_DEBUG=1: device-side checks of every TMA tile's place, the tile
cursors and the workspace indices; see csrc/tc_ptx.cuh). The Python binding
loads it when FLARE_LIBRARY_VARIANT=debug is set in the environment.
"""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libflare.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(BUILD_DEBUG, "libflare.so")


def lib_path(debug: bool = False) -> str:
    return LIB_DEBUG if debug else LIB
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
              "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))


def up_to_date(debug: bool = False) -> bool:
    lib = lib_path(debug)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs() + [os.path.abspath(__file__)])


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile every csrc/*.cu for sm_103a and link libflare.so (the checking
    variant with debug=True); returns its path."""
    lib = lib_path(debug)
    if not force and up_to_date(debug):
        return lib
    out_dir = os.path.dirname(lib)
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    flags = [*extra_flags, "-DFLARE_DEBUG=1"] if debug else list(extra_flags)

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd))
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
