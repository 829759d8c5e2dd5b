"""Builds libmgemm.so in-tree from csrc/ with nvcc for sm_103a.

The translation units compile in parallel (one ``-gencode``), then link into
one shared library beside this file.  The CUDA runtime is linked statically
(nvcc's default), so loading the library needs no GPU; the driver is reached
at run time only.  A rebuild happens when any source is newer than the
library.
"""

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libmgemm.so")

SOURCES = ["args.cu", "quant.cu", "gemm_bf16.cu", "gemm_fp8.cu", "gemm_api.cu", "gemm_f8i4.cu", "gemm_sparse.cu",
           "noalloc.cu",
           "routing.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I" + INCLUDE]


def _nvcc():
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmgemm.so")


def _inputs():
    files = []
    for d in (CSRC, INCLUDE):
        for f in os.listdir(d):
            if f.endswith((".cu", ".cuh", ".h", ".map")):
                files.append(os.path.join(d, f))
    files.append(os.path.abspath(__file__))
    return files


def source_hash():
    """sha256 over the CUDA sources and the header (identifies a kernel build)."""
    import hashlib

    h = hashlib.sha256()
    for f in sorted(_inputs()):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(os.path.basename(f).encode())
            with open(f, "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


# the files that make up the grouped GEMM kernels (a change to any of them
# invalidates counters taken from an earlier build of those kernels)
GEMM_FILES = ["common.cuh", "gemm.cuh", "gemm_launch.cuh", "gemm_bf16.cu", "gemm_fp8.cu", "gemm_api.cu"]


def gemm_source_hash():
    """sha256 over the grouped GEMM's sources and the header."""
    import hashlib

    h = hashlib.sha256()
    for f in GEMM_FILES:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    with open(os.path.join(INCLUDE, "mgemm.h"), "rb") as fh:
        h.update(fh.read())
    return h.hexdigest()[:16]


def up_to_date():
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force=False, verbose=False, extra_flags=()):
    """Compile and link; returns the library path.  Raises on a compiler error."""
    if not force and up_to_date():
        return LIB_PATH
    return _build_into(LIB_PATH, BUILD_DIR, verbose, extra_flags)


def build_variant(name, defines, force=False):
    """A separately named copy of the library (``lib<name>.so`` beside the
    product's), compiled from the same sources with extra preprocessor
    definitions.  Only tests load such a copy (for example one whose pipeline
    waits give up at once, to exercise the timeout path); the binding never
    does."""
    path = os.path.join(PKG, f"lib{name}.so")
    if not force and os.path.exists(path):
        t = os.path.getmtime(path)
        if all(os.path.getmtime(f) <= t for f in _inputs()):
            return path
    flags = [f"-D{k}={v}" for k, v in sorted(defines.items())]
    return _build_into(path, os.path.join(PKG, "_build_" + name), False, flags)


def _build_into(lib_path, build_dir, verbose, extra_flags):
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout, r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + ".tmp"
    # export only the C ABI (exports.map): no C++ symbol of the library can be
    # bound to another copy of it in the same process
    cmd = [nvcc, *ARCH, "-shared", "-Xlinker", "--version-script=" + os.path.join(CSRC, "exports.map"), "-o", tmp,
           *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force=True, verbose=False))
