"""Build libminite.so (the CUDA kernels behind include/minite.h) in-tree.

Compiles every ``csrc/*.cu`` for sm_103a in parallel with nvcc and links a
shared library next to this file. Usage: ``python -m
nvfp4_w4a4_moe_permute_gb300.build`` or ``build()`` from Python.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libminite.so")
ROOT = os.path.dirname(HERE)
BUILD_DIR = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    return r.returncode, r.stdout


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile and link; returns the path of libminite.so. Raises on failure."""
    nvcc = nvcc_path()
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = srcs + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        [os.path.join(ROOT, "include", "minite.h"), os.path.abspath(__file__)]
    if not force and os.path.exists(LIB):
        lib_t = os.path.getmtime(LIB)
        if all(os.path.getmtime(d) <= lib_t for d in deps):
            return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose else []

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
        rc, out = _run([nvcc] + NVCC_FLAGS + extra + ["-c", src, "-o", obj])
        return src, obj, rc, out

    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(compile_one, srcs))
    for src, _, rc, out in results:
        if verbose or rc != 0:
            sys.stderr.write(out)
        if rc != 0:
            raise RuntimeError(f"nvcc failed on {src}")
    objs = [o for _, o, _, _ in results]
    tmp = LIB + ".tmp"
    rc, out = _run([nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs +
                   ["-Xlinker", "-rpath,/usr/local/cuda/lib64"])
    if rc != 0:
        sys.stderr.write(out)
        raise RuntimeError("link of libminite.so failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
