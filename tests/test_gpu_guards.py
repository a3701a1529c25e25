"""Out-of-bounds writes caught without a memory sanitizer.

Two checks, on the tiny fp32 layer and the h1024 Q4_K layer (whole chunks and
ragged lengths):

* guard bytes: every buffer a call writes (outputs, states, conv tails,
  workspaces and scratch) sits between two 4 KB guard regions filled with a
  sentinel byte; after the call every guard byte must be unchanged;
* the debug library (``libgdn_debug.so``, the same kernels compiled with
  GDN_DEBUG): every global store's index is checked against the extent its
  kernel was given, and a failed check skips the store and makes
  gdn_sync_status report GDN_EINDEX.  Its results must equal the release
  library's bit for bit (the checks do not touch the arithmetic).
"""
import ctypes

import numpy as np
import pytest
import torch

from hybrid_gated_deltanet_q4k_gb300 import lib as gl
from hybrid_gated_deltanet_q4k_gb300 import synth
from hybrid_gated_deltanet_q4k_gb300.api import DeviceLayer
from oracle import q4k

from gpu_util import DEV, Guarded, bf16_dev, f16_dev, f32_dev, guarded, stream

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def both_libraries():
    gl.load(build=True)
    return gl.load(debug=True)


def _status_ok(lib):
    assert lib.gdn_sync_status(stream(), check=False) == gl.GDN_OK, lib.last_error()


def _same(a: torch.Tensor, b: torch.Tensor) -> bool:
    if a.dtype in (torch.bfloat16, torch.float16):
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a, b)


def _prefill(spec, layer, tok, n, debug):
    dl = DeviceLayer(spec, layer, debug=debug)
    q4 = spec.wtype == "q4k"
    x = bf16_dev(tok["x_bits"][:n]) if q4 else f32_dev(tok["x"][:n])
    la, bb = f32_dev(tok["log_a"][:n]), f32_dev(tok["b"][:n])
    gs, state = guarded((spec.n_v_heads, spec.dv, spec.dk), torch.float32)
    gc, conv = guarded((spec.c_conv, 3), torch.float32)
    gy, y = guarded((n, spec.hidden), torch.bfloat16 if q4 else torch.float32)
    gw = Guarded(dl.workspace_bytes(n))
    ws = gw.view(torch.uint8, (gw.n,))
    dl.prefill(x, None, state, conv, y, ws, gate_log_a=la, gate_b=bb)
    _status_ok(dl.lib)
    assert all(g.intact() for g in (gs, gc, gy, gw))
    return y.clone(), state.clone(), conv.clone()


@pytest.mark.parametrize("name,n", [("tiny_f32", 64), ("tiny_f32", 37), ("h1024", 512), ("h1024", 130)])
def test_prefill_guards_and_debug_library(name, n):
    spec = synth.SPECS[name]
    layer = synth.make_layer(spec)
    tok = synth.make_tokens(spec, n, seed=n + 500)
    rel = _prefill(spec, layer, tok, n, debug=False)
    dbg = _prefill(spec, layer, tok, n, debug=True)
    assert all(_same(a, b) for a, b in zip(rel, dbg))


@pytest.mark.parametrize("name", ["tiny_f32", "h1024"])
def test_batch_guards_and_debug_library(name):
    spec = synth.SPECS[name]
    layer = synth.make_layer(spec)
    lens = [64, 3, 0, 100]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T, S = int(cu[-1]), len(lens)
    tok = synth.make_tokens(spec, T, seed=31)
    q4 = spec.wtype == "q4k"
    out = []
    for debug in (False, True):
        dl = DeviceLayer(spec, layer, debug=debug)
        x = bf16_dev(tok["x_bits"]) if q4 else f32_dev(tok["x"])
        gs, st = guarded((S, spec.n_v_heads, spec.dv, spec.dk), torch.float32)
        gc, cv = guarded((S, spec.c_conv, 3), torch.float32)
        gy, y = guarded((T, spec.hidden), torch.bfloat16 if q4 else torch.float32)
        gw = Guarded(dl.batch_workspace_bytes(T, S))
        dl.prefill_batch(x, cu, None, st, cv, y, gw.view(torch.uint8, (gw.n,)), gate_log_a=f32_dev(tok["log_a"]),
                         gate_b=f32_dev(tok["b"]))
        _status_ok(dl.lib)
        assert all(g.intact() for g in (gs, gc, gy, gw))
        out.append((y.clone(), st.clone(), cv.clone()))
    assert all(_same(a, b) for a, b in zip(*out))


@pytest.mark.parametrize("name,n", [("h1024", 3), ("h1024", 1), ("tiny_f32", 2)])
def test_decode_guards_and_debug_library(name, n):
    spec = synth.SPECS[name]
    layer = synth.make_layer(spec)
    tok = synth.make_tokens(spec, n, seed=n + 40)
    rng = np.random.default_rng(n)
    st0 = rng.normal(0, 0.3, size=(n, spec.n_v_heads, spec.dv, spec.dk)).astype(np.float32)
    cv0 = rng.normal(0, 1, size=(n, spec.c_conv, 3)).astype(np.float32)
    q4 = spec.wtype == "q4k"
    out = []
    for debug in (False, True):
        dl = DeviceLayer(spec, layer, debug=debug)
        x = bf16_dev(tok["x_bits"]) if q4 else f32_dev(tok["x"])
        gs, st = guarded(st0.shape, torch.float32, torch.from_numpy(st0))
        gc, cv = guarded(cv0.shape, torch.float32, torch.from_numpy(cv0))
        gy, y = guarded((n, spec.hidden), torch.bfloat16 if q4 else torch.float32)
        gw = Guarded(dl.decode_workspace_bytes(n))
        dl.decode(x, st, cv, y, gw.view(torch.uint8, (gw.n,)), gate_log_a=f32_dev(tok["log_a"]), gate_b=f32_dev(tok["b"]))
        _status_ok(dl.lib)
        assert all(g.intact() for g in (gs, gc, gy, gw))
        out.append((y.clone(), st.clone(), cv.clone()))
    assert all(_same(a, b) for a, b in zip(*out))


def _delta_inputs(spec, n, rng):
    hk, hv, d = spec.n_qk_heads, spec.n_v_heads, spec.dk
    q = rng.normal(size=(n, hk, d))
    q = q / np.linalg.norm(q, axis=-1, keepdims=True) * d ** -0.5
    k = rng.normal(size=(n, hk, d))
    k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.normal(size=(n, hv, d))
    qkv = np.concatenate([q.reshape(n, -1), k.reshape(n, -1), v.reshape(n, -1)], axis=1)
    la = -np.logaddexp(0, rng.normal(size=(n, hv)))
    b = 1 / (1 + np.exp(-rng.normal(size=(n, hv))))
    return f16_dev(qkv), f32_dev(la), f32_dev(b)


@pytest.mark.parametrize("name,n", [("tiny_f32", 200), ("h1024", 4200)])
def test_stage_calls_guards_and_debug_library(name, n):
    """Step 1a (Q4_K to int8 rows), step 1b (x quantisation) and step 3 (the
    delta rule with its scratch; 4200 tokens run as two token segments on two
    streams) with guarded outputs, on both libraries."""
    spec = synth.SPECS[name]
    rng = np.random.default_rng(n)
    dev = {k: f32_dev(np.zeros(64, np.float32)) for k in ("w_in", "w_out", "conv_w", "A_log", "dt_bias", "norm_w")}
    s = gl.make_layer_struct(spec, dev)
    qkv, la, b = _delta_inputs(spec, n, rng)
    s0 = f32_dev(rng.normal(0, 0.3, size=(spec.n_v_heads, spec.dv, spec.dk)))
    rows, cols = 300, 1024
    blocks = torch.from_numpy(q4k.pack_q4k(rng.normal(0, 0.02, size=(rows, cols)).astype(np.float32))).to(DEV)
    xq = bf16_dev(synth._to_bf16_bits(rng.normal(size=(rows, cols)).astype(np.float32)))
    out = []
    for debug in (False, True):
        L = gl.load(debug=debug)
        gq, q8 = guarded((rows, cols), torch.int8)
        gsw, sw = guarded((rows,), torch.float32)
        L.q4k_deq_i8(gl.ptr(blocks), rows, cols, gl.ptr(q8), gl.ptr(sw), stream())
        gxc, xc = guarded((rows, cols), torch.float16)
        gsx, sx = guarded((rows,), torch.float32)
        L.gdn_quant_rows(gl.ptr(xq), rows, cols, gl.ptr(xc), gl.ptr(sx), stream())
        go, o = guarded((n, spec.c_v), torch.float16)
        gst, st = guarded((spec.n_v_heads, spec.dv, spec.dk), torch.float32)
        nbytes = L.gdn_delta_rule_scratch_size(ctypes.byref(s), n)
        gsc = Guarded(nbytes)
        L.gdn_delta_rule(ctypes.byref(s), gl.ptr(qkv), gl.ptr(la), gl.ptr(b), n, gl.ptr(s0), gl.ptr(st), gl.ptr(o),
                         gl.ptr(gsc.view(torch.uint8, (nbytes,))), nbytes, stream())
        _status_ok(L)
        assert all(g.intact() for g in (gq, gsw, gxc, gsx, go, gst, gsc))
        out.append((q8.clone(), sw.clone(), xc.clone(), sx.clone(), o.clone(), st.clone()))
    assert all(_same(a, b) for a, b in zip(*out))


def test_attention_guards_and_debug_library():
    rng = np.random.default_rng(3)
    nq, nk, hq, hkv, d = 200, 330, 4, 2, 128
    mk = lambda *sh: bf16_dev(synth._to_bf16_bits(rng.normal(size=sh).astype(np.float32)))  # noqa: E731
    q, k, v = mk(nq, hq, d), mk(nk, hkv, d), mk(nk, hkv, d)
    out = []
    for debug in (False, True):
        L = gl.load(debug=debug)
        go, o = guarded((nq, hq, d), torch.bfloat16)
        nbytes = L.gdn_attn_workspace_size(nk, hkv, d)
        gw = Guarded(nbytes)
        L.gdn_attn_prefill(gl.ptr(q), gl.ptr(k), gl.ptr(v), nq, nk, hq, hkv, d, 0.0, gl.ptr(o),
                           gl.ptr(gw.view(torch.uint8, (nbytes,))), nbytes, stream())
        _status_ok(L)
        assert go.intact() and gw.intact()
        out.append(o.clone())
    assert _same(out[0], out[1])


def test_guard_detects_a_write_past_the_buffer():
    """The guard itself: a copy one element past the view's end changes a guard byte."""
    g, v = guarded((100,), torch.float32)
    assert g.intact()
    g.raw[g.GUARD + g.n: g.GUARD + g.n + 4] = 0
    assert not g.intact()
