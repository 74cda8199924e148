"""Build libfnospec.so in-tree with nvcc for sm_103a.

Each .cu under csrc/ is compiled to an object in parallel, then linked into
fourier_neural_spectral_gb300/libfnospec.so against the shared CUDA runtime.
With --debug the same sources are compiled with -DFNO_DEBUG into
libfnospec_debug.so (every global store of the main kernels range-checked;
loaded instead of the release library when FNO_DEBUG_BOUNDS=1).
Usage: python -m fourier_neural_spectral_gb300.build [--force] [--verbose-ptxas] [--debug]
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
LIB = os.path.join(PKG, "libfnospec.so")
DEBUG_BUILD_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB = os.path.join(PKG, "libfnospec_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libfnospec cannot be built")


def _flags(verbose_ptxas: bool, debug: bool = False) -> list[str]:
    f = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
         "--expt-relaxed-constexpr"] + ARCH
    if debug:
        f += ["-DFNO_DEBUG"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(d) > t for d in _deps())


def build(force: bool = False, verbose_ptxas: bool = False, quiet: bool = True,
          debug: bool = False) -> str:
    lib = DEBUG_LIB if debug else LIB
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    if not force and not verbose_ptxas and not _stale(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    flags = _flags(verbose_ptxas, debug)
    srcs = _sources()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        cmd = [cc, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, (r.stdout + r.stderr)

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(compile_one, srcs))
    logs = "".join(l for _, l in results)
    if verbose_ptxas or not quiet:
        sys.stderr.write(logs)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, "-shared", *ARCH, "-cudart", "shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    ap.add_argument("--debug", action="store_true",
                    help="build the range-checked library libfnospec_debug.so")
    a = ap.parse_args()
    print(build(force=a.force, verbose_ptxas=a.verbose_ptxas, quiet=False, debug=a.debug))
