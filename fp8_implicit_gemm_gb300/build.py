"""Build the CUDA library of this package in-tree: ``_build/libconv3d_fp8.so`` for sm_103a.

nvcc compiles each translation unit in parallel, then links a shared library with the CUDA
runtime linked statically and no link-time dependency on the driver library (the driver entry
point for tensor-map encoding is looked up at run time), so the library also loads on a machine
without a GPU, where only the host-only entry points can do anything useful.

    python -m fp8_implicit_gemm_gb300.build [--force]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
REPO_ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(REPO_ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "libconv3d_fp8.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
SOURCES = ["api.cu", "pack.cu", "conv_tc.cu", "conv_tc_pair.cu", "quant.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                 "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return cand


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)
             if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "conv3d_fp8.h"))
    files.append(os.path.abspath(__file__))
    return files


# The write-counting test build (C3D_COUNT_WRITES): the same sources, every store to y also counted
COUNT_LIB_PATH = os.path.join(BUILD_DIR, "libconv3d_fp8_count.so")


def up_to_date(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build_counting(force: bool = False) -> str:
    """The write-counting build, for tests; returns its path."""
    return build(force=force, extra_flags=["-DC3D_COUNT_WRITES"], out=COUNT_LIB_PATH)


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          out: str = LIB_PATH) -> str:
    """Compile and link; returns the path of the shared library."""
    if not force and up_to_date(out):
        return out
    nvcc = _nvcc()
    obj_dir = os.path.join(BUILD_DIR, "obj" if out == LIB_PATH else "obj_" +
                           os.path.splitext(os.path.basename(out))[0])
    os.makedirs(obj_dir, exist_ok=True)
    flags = CFLAGS + (extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
