"""Build the in-tree CUDA library ``_lib/libgdn.so`` for sm_103a.

Each CUDA translation unit is compiled by nvcc in parallel, the host encoder by
g++, and the objects are linked into one shared library.  Rebuilds only when a
source or header is newer than the library.  No cmake, no torch extension
machinery: the library is a plain C ABI (``include/gdn.h``).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libgdn.so")
INCLUDE = os.path.join(ROOT, "include")

CU_SOURCES = ["k_q4k.cu", "k_q6k.cu", "k_quant.cu", "k_gemm.cu", "k_conv.cu", "k_delta.cu", "k_norm.cu", "k_decode.cu", "k_attn.cu", "streams.cu", "gdn_api.cu"]
CPP_SOURCES = ["kquant_pack.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, f) for f in CU_SOURCES + CPP_SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "gdn.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library; returns its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    cmds = []
    objs = []
    for f in CU_SOURCES:
        obj = os.path.join(OUT_DIR, f + ".o")
        objs.append(obj)
        cmds.append([nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
                     "-I", INCLUDE, "-c", os.path.join(CSRC, f), "-o", obj])
    for f in CPP_SOURCES:
        obj = os.path.join(OUT_DIR, f + ".o")
        objs.append(obj)
        cmds.append(["g++", "-O2", "-fPIC", "-std=c++17", "-ffp-contract=off", "-I", INCLUDE, "-c",
                     os.path.join(CSRC, f), "-o", obj])
    with cf.ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        logs = list(ex.map(_run, cmds))
    if verbose:
        for log in logs:
            sys.stdout.write(log)
    tmp = LIB + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
