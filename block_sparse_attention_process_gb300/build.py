"""Build the CUDA library (libbsa.so) in-tree for sm_103a with nvcc.

Every translation unit under ``csrc/`` is compiled in parallel and linked
into ``_lib/libbsa.so`` next to this file.  No CMake, no torch extension
machinery: the library has a plain C ABI (``include/bsa.h``).

``build(debug=True)`` makes the range-checked variant ``_lib/libbsa_debug.so``
(compiled with ``-DBSA_DEBUG=1``: tensor-memory addresses, computed global
rows and mbarrier phases are checked in the kernels, violations reported in
the device error word); the environment variable
``BSA_LIBRARY_VARIANT=debug`` makes the Python binding load it instead.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(ROOT, "_build", "bsa")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "libbsa.so")
LIB_DEBUG = os.path.join(LIBDIR, "libbsa_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xcompiler", "-fvisibility=hidden"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def build(verbose: bool = False, ptxas_info: bool = False, debug: bool = False) -> str:
    build_dir = BUILD + ("_debug" if debug else "")
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if debug:
        extra += ["-DBSA_DEBUG=1"]
    lib = LIB_DEBUG if debug else LIB

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *FLAGS, *extra, "-I", os.path.join(ROOT, "include"), "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            sys.stdout.write(r.stdout + r.stderr)
        return obj

    srcs = sources()
    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_all(verbose: bool = False) -> None:
    """The release library and the range-checked one, compiled concurrently."""
    with ThreadPoolExecutor(max_workers=2) as ex:
        for f in [ex.submit(build, verbose, False, d) for d in (False, True)]:
            f.result()


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="--ptxas" in sys.argv, debug="--debug" in sys.argv))
