"""The ctypes binding mirrors include/gdn.h: the constants it repeats and the
layout of struct gdn_layer (field offsets and size, as gcc lays the header's
struct out on this machine) agree with the header."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

from hybrid_gated_deltanet_q4k_gb300 import lib as gl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


def _defines():
    out = {}
    for m in re.finditer(r"^#define\s+(GDN_[A-Z0-9_]+)\s+\(?(-?\d+)u?\s*(<<\s*(\d+))?\)?", open(HEADER).read(), re.M):
        v = int(m.group(2))
        if m.group(4):
            v <<= int(m.group(4))
        out[m.group(1)] = v
    return out


def test_constants_match_the_header():
    d = _defines()
    for name in ("GDN_OK", "GDN_EINVAL", "GDN_ENOMEM", "GDN_ECUDA", "GDN_ETIMEOUT", "GDN_ERANGE", "GDN_EINDEX", "GDN_W_Q4K",
                 "GDN_W_F32", "GDN_CHUNK", "GDN_MAX_SEQS", "GDN_N_STAGE_EVENTS", "GDN_NOALLOC_SCRATCH_BYTES"):
        assert name in d, name
        assert getattr(gl, name) == d[name], name


def test_layer_struct_layout_matches_the_header(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    fields = [f for f, _ in gl.GdnLayer._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "gdn.h"\nint main(void) {\n'
                   '  printf("size %zu\\n", sizeof(gdn_layer));\n'
                   + "".join(f'  printf("{f} %zu\\n", offsetof(gdn_layer, {f}));\n' for f in fields)
                   + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-std=c99", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], check=True, capture_output=True,
                                                         text=True).stdout.splitlines())
    assert int(got["size"]) == ctypes.sizeof(gl.GdnLayer)
    for f in fields:
        assert int(got[f]) == getattr(gl.GdnLayer, f).offset, f


def _prototypes():
    text = re.sub(r"/\*.*?\*/", " ", open(HEADER).read(), flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    protos = {}
    for m in re.finditer(r"\b((?:gdn|q4k|q6k)_\w+)\s*\(([^;{}()]*)\)\s*;", text):
        args = m.group(2).strip()
        protos[m.group(1)] = 0 if args in ("", "void") else len(args.split(","))
    return protos


def test_binding_signatures_have_the_header_arity():
    protos = _prototypes()
    assert len(protos) >= 20
    for name, (_, argtypes) in gl._SIGNATURES.items():
        assert name in protos, name
        assert len(argtypes) == protos[name], (name, len(argtypes), protos[name])
