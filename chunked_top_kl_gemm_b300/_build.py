"""Build libkdtopk.so (the C ABI plus its sm_103a kernels) in-tree with nvcc.

    python -m chunked_top_kl_gemm_b300._build          # build if stale
    python -m chunked_top_kl_gemm_b300._build --force  # always rebuild

The library lands next to this file; the Python binding loads it from there.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libkdtopk.so")
SOURCES = ["kd_api.cu", "kd_kernels.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))]
    files.append(os.path.join(INCLUDE, "kd_topk_kl.h"))
    files.append(os.path.abspath(__file__))
    return files


def source_hash() -> str:
    """SHA-256 (first 16 hex digits) of every file the library is built
    from: the CUDA sources, the public header and this build script (its
    flags).  The build compiles it into the library (``kd_build_id``)."""
    h = hashlib.sha256()
    for f in _inputs():
        h.update(os.path.relpath(f, ROOT).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def built_id(path: str = LIB):
    """``kd_build_id()`` of the library at ``path``, asked in a child
    process (this process may already hold another copy loaded), or None
    when it cannot be loaded."""
    if not os.path.exists(path):
        return None
    code = ("import ctypes,sys; L=ctypes.CDLL(sys.argv[1]); "
            "L.kd_build_id.restype=ctypes.c_char_p; print(L.kd_build_id().decode())")
    res = subprocess.run([sys.executable, "-c", code, path], capture_output=True, text=True)
    return res.stdout.strip() if res.returncode == 0 else None


def stale() -> bool:
    """True unless the library exists and was built from the sources as
    they are now (by content, not by file times)."""
    return built_id() != source_hash()


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    if not force and not stale():
        return LIB
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared",
           "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC,
           f"-DKD_BUILD_ID=\"{source_hash()}\"",
           "-o", LIB + ".tmp", *[os.path.join(CSRC, s) for s in SOURCES],
           *extra]
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    if verbose and (res.stdout or res.stderr):
        print(res.stdout + res.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    force = "--force" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []
    print(build(force=force or bool(extra), verbose=True, extra=extra))
