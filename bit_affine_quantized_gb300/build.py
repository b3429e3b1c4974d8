"""Builds libmoe_gb300.so in-tree with nvcc for sm_103a only.

Translation units compile in parallel, then one shared-object link.  The
library is rebuilt when a source or header is newer than it (or `force`).
"""
from __future__ import annotations

import concurrent.futures
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build", "moe")
LIB_DIR = os.path.join(HERE, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libmoe_gb300.so")
SOURCES = ["abi.cu", "router.cu", "ffn.cu", "decode.cu", "prefill.cu", "noalloc.cu", "tail.cu", "head.cu", "offload.cu", "prompt.cu"]
HEADERS = ["common.cuh", "fused.cuh", "kernels.h", "abi_internal.h", "dense.cuh"]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [os.path.join(INCLUDE, "moe.h")]
    return files


def needs_build() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"command failed ({res.returncode}): {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    return res.stdout + res.stderr


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile (if needed) and return the library path."""
    if not force and not needs_build():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    objs = []
    jobs = []
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for s in SOURCES:
            obj = os.path.join(BUILD_DIR, s.replace(".cu", ".o"))
            objs.append(obj)
            cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, s), "-o", obj]
            jobs.append(ex.submit(_run, cmd, verbose))
        logs = [j.result() for j in jobs]
    if ptxas_verbose:
        for s, log in zip(SOURCES, logs):
            print(f"== {s}\n{log}")
    tmp = LIB_PATH + ".tmp"
    _run([NVCC, *ARCH, "-shared", "-o", tmp, *objs], verbose)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="--ptxas-v" in sys.argv))
