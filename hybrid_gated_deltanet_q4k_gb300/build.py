"""Build the in-tree CUDA library ``_lib/libgdn.so`` for sm_103a, and its
debug variant ``_lib/libgdn_debug.so``.

Each CUDA translation unit is compiled by nvcc in parallel, the host encoder by
g++, and the objects are linked into one shared library.  The debug variant is
the same sources compiled with GDN_DEBUG: every kernel checks the indices of
its global stores against the extents it was given and, instead of writing
out of bounds, records the failure for gdn_sync_status (GDN_EINDEX).  Rebuilds
only when a source or header is newer than the library.  No cmake, no torch
extension machinery: the library is a plain C ABI (``include/gdn.h``).
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
DEBUG_DIR = os.path.join(OUT_DIR, "debug")
DEBUG_LIB = os.path.join(OUT_DIR, "libgdn_debug.so")
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


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def _compile_cmds(nvcc: str, out_dir: str, defines: list):
    cmds, objs = [], []
    for f in CU_SOURCES:
        obj = os.path.join(out_dir, f + ".o")
        objs.append(obj)
        cmds.append([nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v", *defines,
                     "-I", INCLUDE, "-c", os.path.join(CSRC, f), "-o", obj])
    for f in CPP_SOURCES:
        obj = os.path.join(out_dir, f + ".o")
        objs.append(obj)
        cmds.append(["g++", "-O2", "-fPIC", "-std=c++17", "-ffp-contract=off", *defines, "-I", INCLUDE, "-c",
                     os.path.join(CSRC, f), "-o", obj])
    return cmds, objs


def build(force: bool = False, verbose: bool = False, debug: bool = True) -> str:
    """Compile and link the library (and, with ``debug``, its debug variant);
    returns the release library's path."""
    targets = [(LIB, OUT_DIR, [])]
    if debug:
        targets.append((DEBUG_LIB, DEBUG_DIR, ["-DGDN_DEBUG"]))
    targets = [t for t in targets if force or not up_to_date(t[0])]
    if not targets:
        return LIB
    nvcc = _nvcc()
    cmds, links = [], []
    for lib, out_dir, defines in targets:
        os.makedirs(out_dir, exist_ok=True)
        c, objs = _compile_cmds(nvcc, out_dir, defines)
        cmds += c
        links.append((lib, objs))
    with cf.ThreadPoolExecutor(max_workers=min(len(cmds), 2 * (os.cpu_count() or 8))) as ex:
        logs = list(ex.map(_run, cmds))
    if verbose:
        for log in logs:
            sys.stdout.write(log)
    for lib, objs in links:
        tmp = lib + ".tmp"
        _run([nvcc, *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
