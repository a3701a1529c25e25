"""End-to-end parity of gdn_prefill with the oracle, plus the session-extend,
ubatching and determinism properties.

End to end the oracle is fed only x, the drawn gates and the packed weights.
The projections are bit-exact, so every difference comes from the
floating-point stages (bf16 activations between stages, fp32 recurrence,
int8 re-quantisation of the gated-norm output).  y must agree within
relative L2 1e-2 (the tolerance for int8 projections: re-quantising o_hat to
int8 amplifies o's rounding), the final state within 2e-3 (the tolerance for
the recurrence with fp32 state: the projections feeding it are bit-exact), the
conv state exactly (it holds raw projection outputs).
"""
import numpy as np
import pytest
import torch

from hybrid_gated_deltanet_q4k_gb300 import synth
from hybrid_gated_deltanet_q4k_gb300.api import DeviceLayer
from oracle import layer as OL

from gpu_util import DEV, bf16_dev, bf16_host_f32, f32_dev, oracle_params, rel_l2

pytestmark = pytest.mark.gpu

Y_TOL = 1e-2        # end to end through two int8 projections
STATE_TOL = 2e-3    # the recurrence with fp32 state


def _x_dev(spec, tok):
    return bf16_dev(tok["x_bits"]) if spec.wtype == "q4k" else f32_dev(tok["x"])


def _y_host(spec, y):
    return bf16_host_f32(y) if spec.wtype == "q4k" else y.cpu().numpy()


def _new_y(spec, n):
    return torch.empty(n, spec.hidden, dtype=torch.bfloat16 if spec.wtype == "q4k" else torch.float32, device=DEV)


def _run(dl, spec, tok, n=None, ws_tokens=None, state=None, conv=None, start=0):
    n = tok["x"].shape[0] - start if n is None else n
    sl = slice(start, start + n)
    x = _x_dev(spec, {k: v[sl] for k, v in tok.items() if k in ("x", "x_bits")})
    la, b = f32_dev(tok["log_a"][sl]), f32_dev(tok["b"][sl])
    if state is None:
        state, conv = dl.new_state()
    y = _new_y(spec, n)
    ws = dl.new_workspace(ws_tokens or n)
    dl.prefill(x, state, state, conv, y, ws, gate_log_a=la, gate_b=b)
    torch.cuda.synchronize()
    return y, state, conv


def _check_vs_oracle(spec, dl, layer, tok, y, state, conv):
    p = oracle_params(spec, layer)
    ref = OL.layer_forward(p, tok["x"], gate_log_a=tok["log_a"], gate_b=tok["b"])
    assert rel_l2(_y_host(spec, y), ref["y"]) <= Y_TOL
    assert rel_l2(state.cpu().numpy(), ref["state"]) <= STATE_TOL
    if spec.wtype == "q4k":
        assert np.array_equal(conv.cpu().numpy(), ref["conv_tail"].astype(np.float32))
    else:
        assert rel_l2(conv.cpu().numpy(), ref["conv_tail"]) <= 2 ** -8
    return ref


@pytest.mark.parametrize("name", ["tiny_f32", "h1024", "h2560"])
def test_prefill_matches_oracle(name):
    spec = synth.SPECS[name]
    layer = synth.make_layer(spec)
    tok = synth.make_tokens(spec, spec.n_tokens, seed=spec.seed + 10)
    dl = DeviceLayer(spec, layer)
    y, state, conv = _run(dl, spec, tok)
    _check_vs_oracle(spec, dl, layer, tok, y, state, conv)


SMALL = synth.LayerSpec("small", 512, 2, 4, 128, 128, 0, "q4k", 11, "softplus_normal")


@pytest.mark.parametrize("n", [1, 2, 3, 63, 65, 127, 513])
def test_prefill_ragged_lengths(n):
    spec = SMALL
    layer = synth.make_layer(spec)
    tok = synth.make_tokens(spec, n, seed=n)
    dl = DeviceLayer(spec, layer)
    y, state, conv = _run(dl, spec, tok)
    _check_vs_oracle(spec, dl, layer, tok, y, state, conv)


def test_prefill_computed_gates():
    """Gates from the beta/alpha projection rows (no drawn gates)."""
    spec = SMALL
    layer = synth.make_layer(spec)
    layer["A_log"] = np.full(spec.n_v_heads, -1.0, np.float32)
    layer["dt_bias"] = np.full(spec.n_v_heads, 0.5, np.float32)
    tok = synth.make_tokens(spec, 100, seed=3)
    dl = DeviceLayer(spec, layer)
    state, conv = dl.new_state()
    y = _new_y(spec, 100)
    ws = dl.new_workspace(100)
    dl.prefill(bf16_dev(tok["x_bits"]), None, state, conv, y, ws)
    torch.cuda.synchronize()
    ref = OL.layer_forward(oracle_params(spec, layer), tok["x"])
    assert rel_l2(bf16_host_f32(y), ref["y"]) <= Y_TOL
    assert rel_l2(state.cpu().numpy(), ref["state"]) <= STATE_TOL


def test_extend_equals_full_prefill_4b_layer():
    """Session extend on the 4B-like layer: 8 sequences, a 2048-token prefix with its
    saved fp32 state and conv tail, then U[1, 4096] more tokens; against a full
    re-prefill of the concatenation.  With the prefix a whole number of chunks
    the two runs do the same arithmetic, so they agree bit for bit."""
    spec = synth.SPECS["extend"]
    layer = synth.make_layer(spec)
    dl = DeviceLayer(spec, layer)
    cases = synth.make_extend_case(spec)
    for i, tok in enumerate(cases):
        n0, m = tok["prefix"], tok["extension"]
        yf, sf, cf_ = _run(dl, spec, tok)
        ya, sa, ca = _run(dl, spec, tok, n=n0)
        yb, sb, cb = _run(dl, spec, tok, start=n0, state=sa, conv=ca)
        assert torch.equal(torch.cat([ya, yb]).view(torch.int16), yf.view(torch.int16))
        assert torch.equal(sb, sf) and torch.equal(cb, cf_)
        if i == 0:   # and against the oracle's re-prefill
            _check_vs_oracle(spec, dl, layer, tok, yf, sf, cf_)


@pytest.mark.parametrize("n0", [1, 37, 100])
def test_extend_at_odd_boundaries(n0):
    spec = SMALL
    layer = synth.make_layer(spec)
    dl = DeviceLayer(spec, layer)
    tok = synth.make_tokens(spec, 300, seed=n0)
    yf, sf, cf_ = _run(dl, spec, tok)
    ya, sa, ca = _run(dl, spec, tok, n=n0)
    yb, sb, cb = _run(dl, spec, tok, start=n0, state=sa, conv=ca)
    # both runs are within tolerance of the exact layer; they differ by the rounding of
    # the fp16 chunk products at different chunk boundaries (state: recurrence bound;
    # y: the end-to-end int8 bound, since re-quantising o_hat amplifies o's rounding)
    y2 = torch.cat([ya, yb])
    assert rel_l2(bf16_host_f32(y2), bf16_host_f32(yf)) <= 1e-2
    assert rel_l2(sb.cpu().numpy(), sf.cpu().numpy()) <= 2e-3
    assert torch.equal(cb, cf_)


def test_ubatched_workspace_is_bit_identical():
    """A workspace holding fewer tokens than N runs in passes; with passes of whole
    chunks the result is the same bits as one pass."""
    spec = synth.SPECS["h1024"]
    layer = synth.make_layer(spec)
    dl = DeviceLayer(spec, layer)
    tok = synth.make_tokens(spec, 700, seed=4)
    y1, s1, c1 = _run(dl, spec, tok)
    y2, s2, c2 = _run(dl, spec, tok, ws_tokens=128)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(s1, s2) and torch.equal(c1, c2)
    y3, s3, c3 = _run(dl, spec, tok, ws_tokens=1)    # one token per pass
    assert rel_l2(bf16_host_f32(y3), bf16_host_f32(y1)) <= 1e-2
    assert rel_l2(s3.cpu().numpy(), s1.cpu().numpy()) <= 2e-3


def test_runs_are_deterministic():
    spec = synth.SPECS["h2560"]
    layer = synth.make_layer(spec)
    dl = DeviceLayer(spec, layer)
    tok = synth.make_tokens(spec, 1000, seed=5)
    y1, s1, _ = _run(dl, spec, tok)
    y2, s2, _ = _run(dl, spec, tok)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)) and torch.equal(s1, s2)


def test_errors_are_statuses_not_fallbacks():
    spec = SMALL
    dl = DeviceLayer(spec, synth.make_layer(spec))
    tok = synth.make_tokens(spec, 10, seed=1)
    state, conv = dl.new_state()
    y = _new_y(spec, 10)
    small = torch.empty(dl.workspace_bytes(1) - 4096, dtype=torch.uint8, device=DEV)
    assert dl.prefill(bf16_dev(tok["x_bits"]), None, state, conv, y, small, check=False) == -2
    ws = dl.new_workspace(10)
    assert dl.prefill(bf16_dev(tok["x_bits"])[:0], None, state, conv, y, ws, check=False) == -1


def _stage_by_stage(dl, spec, x, la, bb, state_in, conv_state):
    """The layer through the stage entry points one by one (the conv as its own
    kernel on the projection's bf16 output); returns y, the state and the conv
    state.  la, bb = None: gates computed from the projection."""
    import ctypes

    from hybrid_gated_deltanet_q4k_gb300 import lib as gl

    L = dl.lib
    n, H, hv = x.shape[0], spec.hidden, spec.n_v_heads
    c_v, c_conv, r_in = spec.c_v, spec.c_conv, spec.r_in
    nbf = spec.c_conv + spec.c_v
    s = dl.struct(la, bb)
    sp = ctypes.byref(s)
    st = gl.stream_handle()
    wc_in = torch.empty(r_in, H, dtype=torch.float16, device=DEV)
    ws_in = torch.empty(r_in, dtype=torch.float32, device=DEV)
    wc_out = torch.empty(H, c_v, dtype=torch.float16, device=DEV)
    ws_out = torch.empty(H, dtype=torch.float32, device=DEV)
    L.gdn_q4k_deq_codes(gl.ptr(dl.dev["w_in"]), r_in, H, gl.ptr(wc_in), gl.ptr(ws_in), st)
    L.gdn_q4k_deq_codes(gl.ptr(dl.dev["w_out"]), H, c_v, gl.ptr(wc_out), gl.ptr(ws_out), st)
    xc = torch.empty(n, H, dtype=torch.float16, device=DEV)
    sx = torch.empty(n, dtype=torch.float32, device=DEV)
    L.gdn_quant_rows(gl.ptr(x), n, H, gl.ptr(xc), gl.ptr(sx), st)
    qkvz = torch.empty(n, nbf, dtype=torch.bfloat16, device=DEV)
    ba = torch.empty(n, 2 * hv, dtype=torch.float32, device=DEV)
    L.gdn_gemm_codes(gl.ptr(xc), gl.ptr(sx), gl.ptr(wc_in), gl.ptr(ws_in), n, r_in, H, gl.ptr(qkvz), nbf, nbf,
                     gl.ptr(ba), 2 * hv, st)
    qkv = torch.empty(n, c_conv, dtype=torch.float16, device=DEV)
    la_c = torch.empty(n, hv, dtype=torch.float32, device=DEV)
    b_c = torch.empty(n, hv, dtype=torch.float32, device=DEV)
    L.gdn_conv(sp, gl.ptr(qkvz), nbf, n, gl.ptr(conv_state), gl.ptr(ba), 2 * hv, gl.ptr(qkv), gl.ptr(la_c),
               gl.ptr(b_c), st)
    L.gdn_conv_state_update(sp, gl.ptr(qkvz), nbf, n, gl.ptr(conv_state), st)
    nbytes = L.gdn_delta_rule_scratch_size(sp, n)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    state = torch.empty_like(state_in)
    o = torch.empty(n, c_v, dtype=torch.float16, device=DEV)
    ga, gb = (la, bb) if la is not None else (la_c, b_c)
    L.gdn_delta_rule(sp, gl.ptr(qkv), gl.ptr(ga), gl.ptr(gb), n, gl.ptr(state_in), gl.ptr(state), gl.ptr(o),
                     gl.ptr(scratch), nbytes, st)
    oc = torch.empty(n, c_v, dtype=torch.float16, device=DEV)
    so = torch.empty(n, dtype=torch.float32, device=DEV)
    z = qkvz[:, c_conv:]
    L.gdn_gated_norm(sp, gl.ptr(o), gl.ptr(z), nbf, n, gl.ptr(oc), gl.ptr(so), 0, st)
    y = torch.empty(n, H, dtype=torch.bfloat16, device=DEV)
    L.gdn_gemm_codes(gl.ptr(oc), gl.ptr(so), gl.ptr(wc_out), gl.ptr(ws_out), n, H, c_v, gl.ptr(y), H, H, 0, 0, st)
    torch.cuda.synchronize()
    return y, state, conv_state


@pytest.mark.parametrize("n", [1, 2, 3, 4, 127, 128, 130, 300, 515])
@pytest.mark.parametrize("gates", ["drawn", "computed"])
def test_prefill_equals_stage_calls(n, gates):
    """gdn_prefill chains the step kernels inside one call (dequant, x
    quantisation, projection, conv, delta rule with its prep on a second
    stream, gated norm, output projection).  It must give the same bits as the
    stage entry points called one by one: for lengths around the chunk and
    tile boundaries, a nonzero initial conv state (not bf16-exact), drawn and
    computed gates."""
    spec = SMALL
    layer = synth.make_layer(spec)
    tok = synth.make_tokens(spec, n, seed=40 + n)
    dl = DeviceLayer(spec, layer)
    rng = np.random.default_rng(n)
    x = _x_dev(spec, tok)
    la, bb = (f32_dev(tok["log_a"]), f32_dev(tok["b"])) if gates == "drawn" else (None, None)
    s0 = f32_dev(rng.normal(0, 0.3, size=(spec.n_v_heads, spec.dv, spec.dk)))
    c0 = f32_dev(rng.normal(0, 1.0, size=(spec.c_conv, 3)))
    state, conv = s0.clone(), c0.clone()
    y = _new_y(spec, n)
    ws = dl.new_workspace(n)
    dl.prefill(x, state, state, conv, y, ws, gate_log_a=la, gate_b=bb)
    torch.cuda.synchronize()
    y2, state2, conv2 = _stage_by_stage(dl, spec, x, la, bb, s0, c0.clone())
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(state, state2)
    assert torch.equal(conv, conv2)


def _pinned(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.view(dtype) if dtype is not None else t).pin_memory()


# passes of B (first and last B/4) for B = 256 and 128; ramped passes B/8, 3B/8,
# B, ..., 3B/8, B/8 for B = 1024, and with a ragged tail for B = 512
@pytest.mark.parametrize("name,n,pass_tokens", [("h2560", 1000, 256), ("h2560", 4096, 1024), ("tiny_f32", 64, 0),
                                                ("h1024", 513, 128), ("h1024", 2085, 512)])
def test_prefill_host_equals_device_prefill(name, n, pass_tokens):
    """gdn_prefill_host (pinned host x, y and gates, copies overlapped with the
    passes) gives bit for bit what gdn_prefill gives with passes of the same
    size, and stays within the oracle's tolerance."""
    spec = synth.SPECS[name]
    layer = synth.make_layer(spec)
    tok = synth.make_tokens(spec, n, seed=spec.seed + 30)
    dl = DeviceLayer(spec, layer)
    B = pass_tokens or n
    yd, sd, cd = _run(dl, spec, tok, ws_tokens=B)
    q4k = spec.wtype == "q4k"
    xh = _pinned(tok["x_bits"].view(np.int16)) if q4k else _pinned(tok["x"].astype(np.float32))
    yh = torch.empty(n, spec.hidden, dtype=torch.int16 if q4k else torch.float32).pin_memory()
    lah, bh = _pinned(tok["log_a"].astype(np.float32)), _pinned(tok["b"].astype(np.float32))
    state, conv = dl.new_state()
    ws = dl.new_host_workspace(B, gates=True)
    for _ in range(2):     # a second call reuses the copy streams, events and staging slots
        state.zero_()
        conv.zero_()
        yh.zero_()
        dl.prefill_host(xh, None, state, conv, yh, ws, pass_tokens=pass_tokens, gate_log_a=lah, gate_b=bh)
        torch.cuda.current_stream().synchronize()
        yv = yh.view(torch.int16) if q4k else yh
        assert torch.equal(yv, yd.cpu().view(torch.int16) if q4k else yd.cpu())
        assert torch.equal(state, sd) and torch.equal(conv, cd)
    if n <= 1024:
        yy = synth.bf16_bits_to_f32(yh.numpy().view(np.uint16)) if q4k else yh.numpy()
        ref = OL.layer_forward(oracle_params(spec, layer), tok["x"], gate_log_a=tok["log_a"], gate_b=tok["b"])
        assert rel_l2(yy, ref["y"]) <= Y_TOL


def test_prefill_host_computed_gates_and_extend():
    """Without drawn gates, and extending a saved state: two host-fed calls
    (2 passes, then 3) equal one device call over the concatenation."""
    spec = SMALL
    layer = synth.make_layer(spec)
    tok = synth.make_tokens(spec, 640, seed=21)
    dl = DeviceLayer(spec, layer)
    state, conv = dl.new_state()
    y = _new_y(spec, 640)
    dl.prefill(bf16_dev(tok["x_bits"]), None, state, conv, y, dl.new_workspace(128))
    xh = _pinned(tok["x_bits"].view(np.int16))
    yh = torch.empty(640, spec.hidden, dtype=torch.int16).pin_memory()
    s2, c2 = dl.new_state()
    ws = dl.new_host_workspace(128)
    dl.prefill_host(xh[:256], None, s2, c2, yh[:256], ws, pass_tokens=128)
    dl.prefill_host(xh[256:], s2, s2, c2, yh[256:], ws, pass_tokens=128)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(yh, y.cpu().view(torch.int16))
    assert torch.equal(s2, state) and torch.equal(c2, conv)


def test_prefill_host_rejects_pageable_memory():
    from hybrid_gated_deltanet_q4k_gb300 import lib as gl
    spec = SMALL
    layer = synth.make_layer(spec)
    dl = DeviceLayer(spec, layer)
    state, conv = dl.new_state()
    xh = torch.zeros(64, spec.hidden, dtype=torch.int16)          # pageable
    yh = torch.zeros(64, spec.hidden, dtype=torch.int16).pin_memory()
    ws = dl.new_host_workspace(64)
    r = dl.prefill_host(xh, None, state, conv, yh, ws, check=False)
    assert r == gl.GDN_EINVAL and "page-locked" in dl.lib.last_error()
    r = dl.prefill_host(yh, None, state, conv, yh, ws[: dl.host_workspace_bytes(1) - 256], check=False)
    assert r == gl.GDN_ENOMEM


@pytest.mark.parametrize("q6k", [("w_out",), ("w_in", "w_out"), ("w_in",)])
def test_prefill_with_q6k_matrices(q6k):
    """Q4_K_M files hold some matrices in Q6_K: the layer decodes each from its
    own format and matches the oracle doing the same."""
    spec = SMALL
    layer = synth.make_layer(spec)
    tok = synth.make_tokens(spec, 200, seed=len(q6k) + 50)
    dl = DeviceLayer(spec, layer, q6k=q6k)
    y, state, conv = _run(dl, spec, tok)
    p = oracle_params(spec, layer)
    from oracle import q6k as O6
    for name in q6k:
        p[name] = O6.pack_q6k(layer[name])
        p[name + "_fmt"] = "q6k"
        assert np.array_equal(dl.host_blocks[name], p[name])
    ref = OL.layer_forward(p, tok["x"], gate_log_a=tok["log_a"], gate_b=tok["b"])
    assert rel_l2(_y_host(spec, y), ref["y"]) <= Y_TOL
    assert rel_l2(state.cpu().numpy(), ref["state"]) <= STATE_TOL
