"""Build the CUDA library (csrc/*.cu -> _build/libmoe_gb300.so) for sm_103a.

Every translation unit is compiled in parallel with one -gencode
(compute_103a / sm_103a) and linked into a shared library with the static
CUDA runtime; nothing is installed outside this folder.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
# MOE_BUILD_DIR / MOE_NVCC_DEFINES build a variant elsewhere (for example
# with -DMOE_TRACE); MOE_LIBRARY makes the binding load a given build.
BUILD = os.environ.get("MOE_BUILD_DIR", os.path.join(HERE, "_build"))
LIBRARY = os.environ.get("MOE_LIBRARY", os.path.join(BUILD, "libmoe_gb300.so"))
DEFINES = os.environ.get("MOE_NVCC_DEFINES", "").split()
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", os.path.join(ROOT, "include")]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _dependencies():
    deps = _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    return deps + [os.path.join(ROOT, "include", "moe.h")]


def up_to_date() -> bool:
    if not os.path.exists(LIBRARY):
        return False
    built = os.path.getmtime(LIBRARY)
    return all(os.path.getmtime(d) <= built for d in _dependencies())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIBRARY
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose else []

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [NVCC, *ARCH, *FLAGS, *DEFINES, *extra, "-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{res.stderr}")
        if verbose and res.stderr:
            print(res.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(_sources())) as pool:
        objects = list(pool.map(compile_one, _sources()))
    tmp = LIBRARY + f".{os.getpid()}.tmp"
    cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *objects]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stderr}")
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    import sys

    print(build(force=True, verbose="-v" in sys.argv))
