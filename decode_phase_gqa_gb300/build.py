"""Build the in-tree CUDA library ``_build/libkvattn.so`` for sm_103a.

Plain nvcc, no torch extension: the translation units under ``csrc/`` are
compiled in parallel and linked into one shared library (CUDA runtime linked
statically) that the ctypes binding loads.  Rebuilds only what is stale.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libkvattn.so")
HEADER = os.path.join(ROOT, "include", "kvattn.h")

SOURCES = ["kvattn_api.cu", "decode_bf16.cu", "decode_int8.cu", "decode_bf16_layers.cu",
           "decode_int8_layers.cu", "kvattn_noalloc.cu", "combine.cu", "prefill.cu",
           "prefill_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-Wall", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (needed to build the CUDA library)")


def _deps_mtime() -> float:
    paths = [HEADER] + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    return max(os.path.getmtime(p) for p in paths)


def _compile(src: str, nvcc: str, extra, verbose: bool, build_dir: str) -> str:
    obj = os.path.join(build_dir, src.replace(".cu", ".o"))
    srcp = os.path.join(CSRC, src)
    if (os.path.exists(obj) and os.path.getmtime(obj) >= os.path.getmtime(srcp)
            and os.path.getmtime(obj) >= _deps_mtime()):
        return obj
    cmd = [nvcc] + NVCC_FLAGS + list(extra) + ["-c", srcp, "-o", obj + ".tmp"]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    os.replace(obj + ".tmp", obj)
    return obj


def build(force: bool = False, verbose: bool = False, extra_flags=(), variant: str = None) -> str:
    """Compile and link the library; returns its path.

    ``variant``: a named build with ``extra_flags`` (e.g. a test-only macro),
    kept apart in ``_build/<variant>/`` so it never replaces the library."""
    build_dir = BUILD if variant is None else os.path.join(BUILD, variant)
    lib = os.path.join(build_dir, "libkvattn.so")
    os.makedirs(build_dir, exist_ok=True)
    if force:
        for f in os.listdir(build_dir):
            if f.endswith((".o", ".so")):
                os.remove(os.path.join(build_dir, f))
    nvcc = _nvcc()
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, nvcc, extra_flags, verbose, build_dir), SOURCES))
    if not os.path.exists(lib) or any(os.path.getmtime(o) > os.path.getmtime(lib) for o in objs):
        cmd = [nvcc] + ARCH + ["-shared", "-o", lib + ".tmp"] + objs
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(lib + ".tmp", lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True))
