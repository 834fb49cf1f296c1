"""Builds libtpmlp.so (the C-ABI library) from csrc/ with nvcc for sm_103a.

Each .cu file is compiled to an object in parallel, then the objects are
linked into a shared library next to this file. The CUDA runtime is linked
statically, so loading the library needs no GPU. With debug=True (--debug)
the same sources are compiled with TPMLP_DEBUG defined, which adds the
device-side index checks, into libtpmlp_debug.so (objects under
_build/debug). Usage:

    python -m tensor_transformer_mlp_column_gb300.build_lib [--force] [--ptxas-verbose] [--debug]
"""

from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
REPO_DIR = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(REPO_DIR, "include")
BUILD_DIR = os.path.join(REPO_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libtpmlp.so")
DEBUG_LIB_PATH = os.path.join(PKG_DIR, "libtpmlp_debug.so")
SOURCES = ["api.cu", "gemm_tc.cu", "gemm_pair.cu", "gemm_dual.cu", "gemm_fwd.cu", "simt.cu", "elementwise.cu", "block.cu", "attention.cu", "attn_api.cu", "noalloc.cu", "trace.cu"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in [os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"]:
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "tpmlp.h"))
    files.append(os.path.abspath(__file__))
    return files


def _up_to_date(lib_path: str) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = False, debug: bool = False) -> str:
    """Compile and link libtpmlp.so (libtpmlp_debug.so with debug=True) if
    any source is newer; return its path."""
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    build_dir = os.path.join(BUILD_DIR, "debug") if debug else BUILD_DIR
    if not force and not ptxas_verbose and _up_to_date(lib_path):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    common = ARCH + [
        "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
        "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC,
    ]
    if debug:
        common += ["-DTPMLP_DEBUG=1"]
    if ptxas_verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src: str):
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [nvcc] + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    for src, _, r in results:
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if (ptxas_verbose or r.stderr.strip()) and not quiet:
            sys.stderr.write(r.stderr)
    tmp = lib_path + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [obj for _, obj, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    path = build(force="--force" in sys.argv, ptxas_verbose="--ptxas-verbose" in sys.argv, debug="--debug" in sys.argv)
    print(path)
