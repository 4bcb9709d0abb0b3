"""Build step of libdllm.so: nvcc for sm_103a, in-tree.

``python -m partial_attention_saliency_b300.build`` (or ``build_library()``)
compiles every ``csrc/*.cu`` to an object under ``_build/`` and links them into
``partial_attention_saliency_b300/libdllm.so``.  Objects are rebuilt when their
source, a header or the flags change.
"""
from __future__ import annotations

import glob
import hashlib
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libdllm.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdllm.so")


def _headers_digest() -> str:
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                    + glob.glob(os.path.join(INCLUDE, "*.h"))):
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(NVCC_FLAGS).encode())
    return h.hexdigest()[:16]


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"command failed ({res.returncode}): {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    if verbose and (res.stdout.strip() or res.stderr.strip()):
        print(res.stdout + res.stderr, flush=True)
    return res


def build_library(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile and link libdllm.so; returns its path."""
    nvcc = nvcc_path()
    os.makedirs(BUILD_DIR, exist_ok=True)
    digest = _headers_digest() + hashlib.sha256(" ".join(extra_flags).encode()).hexdigest()[:8]
    objs = []
    changed = force or not os.path.exists(LIB_PATH)
    for src in sorted(glob.glob(os.path.join(CSRC, "*.cu"))):
        with open(src, "rb") as f:
            tag = hashlib.sha256(f.read()).hexdigest()[:16]
        obj = os.path.join(BUILD_DIR, f"{os.path.basename(src)}.{tag}.{digest}.o")
        if force or not os.path.exists(obj):
            _run([nvcc, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj], verbose)
            changed = True
        objs.append(obj)
    if changed or os.path.getmtime(LIB_PATH) < max(os.path.getmtime(o) for o in objs):
        tmp = LIB_PATH + ".tmp"
        _run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], verbose)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    path = build_library(force="--force" in sys.argv, verbose=True)
    print(path)
