"""gdn_prefill_batch: several independent sequences of different lengths in one
call, each with its own recurrent state and conv tail.

Every sequence is chunked from its own first token and the projections are
row-independent, so the batch must give, bit for bit, what gdn_prefill gives
on each sequence alone; the session-extend workload (8 sequences with saved
states, extended by U[1, 4096] tokens) must equal a re-prefill of the whole
prompts, and the oracle bounds one sequence end to end.
"""
import numpy as np
import pytest
import torch

from hybrid_gated_deltanet_q4k_gb300 import lib as gl
from hybrid_gated_deltanet_q4k_gb300 import synth
from hybrid_gated_deltanet_q4k_gb300.api import DeviceLayer
from oracle import layer as OL

from gpu_util import DEV, bf16_dev, bf16_host_f32, f32_dev, oracle_params, rel_l2

pytestmark = pytest.mark.gpu

SMALL = synth.LayerSpec("small", 512, 2, 4, 128, 128, 0, "q4k", 11, "softplus_normal")


def _x(spec, tok):
    return bf16_dev(tok["x_bits"]) if spec.wtype == "q4k" else f32_dev(tok["x"])


def _ydtype(spec):
    return torch.bfloat16 if spec.wtype == "q4k" else torch.float32


def _same(a, b):
    if a.dtype == torch.bfloat16:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a, b)


def _random_states(spec, n_seqs, seed):
    rng = np.random.default_rng(seed)
    st = (0.05 * rng.standard_normal((n_seqs, spec.n_v_heads, spec.dv, spec.dk))).astype(np.float32)
    cv = rng.standard_normal((n_seqs, spec.c_conv, 3)).astype(np.float32)
    return torch.from_numpy(st).to(DEV), torch.from_numpy(cv).to(DEV)


def _per_sequence(dl, spec, tok, cu, state0, conv0, gates):
    """gdn_prefill on each sequence alone: y [T][H], states, conv tails."""
    T = cu[-1]
    y = torch.empty(T, spec.hidden, dtype=_ydtype(spec), device=DEV)
    states, convs = state0.clone(), conv0.clone()
    for i in range(len(cu) - 1):
        a, b = cu[i], cu[i + 1]
        if a == b:
            continue
        sl = slice(a, b)
        x = _x(spec, {k: v[sl] for k, v in tok.items() if k in ("x", "x_bits")})
        la = f32_dev(tok["log_a"][sl]) if gates else None
        bb = f32_dev(tok["b"][sl]) if gates else None
        ws = dl.new_workspace(b - a)
        dl.prefill(x, states[i], states[i], convs[i], y[a:b], ws, gate_log_a=la, gate_b=bb)
    torch.cuda.synchronize()
    return y, states, convs


def _batch(dl, spec, tok, cu, state0, conv0, gates, state_in_null=False):
    T = cu[-1]
    n = len(cu) - 1
    x = _x(spec, tok) if T else None
    y = torch.empty(max(T, 1), spec.hidden, dtype=_ydtype(spec), device=DEV)
    states, convs = state0.clone(), conv0.clone()
    la = f32_dev(tok["log_a"]) if gates else None
    bb = f32_dev(tok["b"]) if gates else None
    ws = dl.new_batch_workspace(T, n)
    dl.prefill_batch(x, cu, None if state_in_null else states, states, convs, y, ws, gate_log_a=la, gate_b=bb)
    torch.cuda.synchronize()
    return y[:T], states, convs


@pytest.mark.parametrize("lens,gates", [
    ([1, 63, 64, 65, 200, 0, 700], True),
    ([5000, 130, 0, 3000, 1], True),        # token segments (rounds) with sequences ending in different ones
    ([300, 17, 129], False),                # gates from the projection
    # the maximum number of sequences, ragged lengths 0..39
    ([int(v) for v in np.random.default_rng(256).integers(0, 40, gl.GDN_MAX_SEQS)], True),
])
def test_batch_equals_each_sequence_alone(lens, gates):
    spec = SMALL
    layer = synth.make_layer(spec)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    tok = synth.make_tokens(spec, int(cu[-1]), seed=len(lens) + 40)
    dl = DeviceLayer(spec, layer)
    s0, c0 = _random_states(spec, len(lens), seed=len(lens))
    yr, sr, cr = _per_sequence(dl, spec, tok, cu, s0, c0, gates)
    yb, sb, cb = _batch(dl, spec, tok, cu, s0, c0, gates)
    assert _same(yb, yr)
    assert torch.equal(sb, sr) and torch.equal(cb, cr)
    assert torch.equal(sb[lens.index(0)], s0[lens.index(0)]) if 0 in lens else True


def test_batch_zero_state_and_tiny_f32_layer():
    spec = synth.SPECS["tiny_f32"]
    layer = synth.make_layer(spec)
    lens = [64, 3, 0, 100]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    tok = synth.make_tokens(spec, int(cu[-1]), seed=5)
    dl = DeviceLayer(spec, layer)
    z_s = torch.zeros(len(lens), spec.n_v_heads, spec.dv, spec.dk, device=DEV)
    z_c = torch.zeros(len(lens), spec.c_conv, 3, device=DEV)
    s_nan = torch.full_like(z_s, float("nan"))        # state_in NULL: state_out is written, never read
    yr, sr, cr = _per_sequence(dl, spec, tok, cu, z_s, z_c, True)
    yb, sb, cb = _batch(dl, spec, tok, cu, s_nan, z_c, True, state_in_null=True)
    assert _same(yb, yr) and torch.equal(sb, sr) and torch.equal(cb, cr)
    assert torch.equal(sb[2], z_s[2])                   # the empty sequence: zero state
    p = oracle_params(spec, layer)
    a, b = cu[3], cu[4]
    ref = OL.layer_forward(p, tok["x"][a:b], gate_log_a=tok["log_a"][a:b], gate_b=tok["b"][a:b])
    assert rel_l2(yb[a:b].cpu().numpy(), ref["y"]) <= 1e-2
    assert rel_l2(sb[3].cpu().numpy(), ref["state"]) <= 2e-3   # recurrence tolerance


def test_batch_session_extend_4b_layer():
    """Session extend on the 4B-like layer, batched: the 8 prefixes of 2048
    tokens in one call from zero state, then the 8 extensions (U[1, 4096]
    tokens each) in one call from the saved states and conv tails.  Both equal
    a full re-prefill of each concatenated prompt bit for bit (the prefix is a
    whole number of chunks), and the first sequence is within the oracle's
    tolerance."""
    spec = synth.SPECS["extend"]
    layer = synth.make_layer(spec)
    dl = DeviceLayer(spec, layer)
    cases = synth.make_extend_case(spec)
    n = len(cases)
    pre = [c["prefix"] for c in cases]
    ext = [c["extension"] for c in cases]
    cat = lambda key, part: np.concatenate(  # noqa: E731
        [c[key][: c["prefix"]] if part == 0 else c[key][c["prefix"]:] for c in cases])
    cu0 = np.concatenate([[0], np.cumsum(pre)]).astype(np.int64)
    cu1 = np.concatenate([[0], np.cumsum(ext)]).astype(np.int64)
    tok0 = {k: cat(k, 0) for k in ("x", "x_bits", "log_a", "b")}
    tok1 = {k: cat(k, 1) for k in ("x", "x_bits", "log_a", "b")}
    s0, c0 = dl.new_batch_state(n)
    _, s1, cv1 = _batch(dl, spec, tok0, cu0, s0, c0, True)
    y2, s2, cv2 = _batch(dl, spec, tok1, cu1, s1, cv1, True)
    for i, c in enumerate(cases):
        full = {k: c[k] for k in ("x", "x_bits", "log_a", "b")}
        cu = np.array([0, c["prefix"] + c["extension"]], np.int64)
        yf, sf, cf = _per_sequence(dl, spec, full, cu, s0[:1], c0[:1], True)
        assert _same(y2[cu1[i]:cu1[i + 1]], yf[c["prefix"]:]), i
        assert torch.equal(s2[i], sf[0]) and torch.equal(cv2[i], cf[0]), i
    c = cases[0]
    ref = OL.layer_forward(oracle_params(spec, layer), c["x"], gate_log_a=c["log_a"], gate_b=c["b"])
    assert rel_l2(bf16_host_f32(y2[: ext[0]]), ref["y"][c["prefix"]:]) <= 1e-2
    assert rel_l2(s2[0].cpu().numpy(), ref["state"]) <= 2e-3   # recurrence tolerance


def test_batch_argument_checks():
    spec = SMALL
    layer = synth.make_layer(spec)
    dl = DeviceLayer(spec, layer)
    s, c = dl.new_batch_state(2)
    x = torch.zeros(10, spec.hidden, dtype=torch.bfloat16, device=DEV)
    y = torch.empty_like(x)
    ws = dl.new_batch_workspace(10, 2)
    bad = [([0, 5, 3], gl.GDN_EINVAL), ([1, 5, 10], gl.GDN_EINVAL)]
    for cu, code in bad:
        assert dl.prefill_batch(x, cu, s, s, c, y, ws, check=False) == code
    assert dl.prefill_batch(x, [0, 5, 10], s, s, c, y, ws[:1024], check=False) == gl.GDN_ENOMEM
    big = list(range(gl.GDN_MAX_SEQS + 2))
    assert dl.prefill_batch(x, big, s, s, c, y, ws, check=False) == gl.GDN_EINVAL
    assert dl.batch_workspace_bytes(10, gl.GDN_MAX_SEQS + 1) == 0
