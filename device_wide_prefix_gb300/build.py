"""Build libdwp.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each .cu under csrc/ compiles to an object in parallel, then one link step
makes device_wide_prefix_gb300/libdwp.so against the shared CUDA runtime.
Host code is portable C++17 (no architecture-specific flags), so the same
sources build on x86_64 and aarch64 hosts.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdwp.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdwp.so")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    pats = ("*.cu", "*.cuh", "*.h")
    files = [f for p in pats for f in glob.glob(os.path.join(CSRC, p))]
    return files + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def compile_flags(extra: list[str] | None = None) -> list[str]:
    return ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC",
            "-Xcompiler", "-Wall", "-I", INCLUDE, "-I", CSRC, *(extra or [])]


def build(force: bool = False, extra: list[str] | None = None, lib: str = LIB,
          verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link; returns the library path.  Raises on a compiler error."""
    if not force and not extra and lib == LIB and up_to_date(lib):
        return lib
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    flags = compile_flags(extra) + (["-Xptxas", "-v"] if ptxas_info else [])
    tag = "" if lib == LIB else "_" + os.path.basename(lib).replace(".so", "")

    def one(src: str) -> str:
        obj = os.path.join(BUILD_DIR, os.path.basename(src).replace(".cu", tag + ".o"))
        cmd = [cc, *flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s%s" % (src, r.stdout, r.stderr))
        if ptxas_info or verbose:
            print(r.stdout + r.stderr, flush=True)
        return obj

    srcs = sources()
    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(one, srcs))
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [cc, "-shared", *ARCH, "-cudart", "shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                ptxas_info="--ptxas" in sys.argv))
