"""Pins for the oracle's conv, norms, gates, gated delta rule and whole layer."""
import math

import numpy as np
import pytest

from oracle import layer as L
from oracle import q4k

from hybrid_gated_deltanet_q4k_gb300 import synth


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


# ----------------------------------------------------------------- elementwise

def test_elementwise_closed_forms():
    assert L.softplus(0.0) == pytest.approx(math.log(2.0), abs=1e-15)
    assert L.softplus(50.0) == pytest.approx(50.0, abs=1e-15)
    assert L.softplus(-50.0) == pytest.approx(math.exp(-50.0), rel=1e-12)
    assert L.sigmoid(0.0) == 0.5
    assert L.silu(0.0) == 0.0
    assert L.silu(30.0) == pytest.approx(30.0, rel=1e-12)
    assert L.silu(-1.0) == pytest.approx(-1.0 / (1.0 + math.e), rel=1e-15)
    # with A_log = dt_bias = 0: a = exp(-softplus(alpha)) = sigmoid(-alpha)
    alpha = np.linspace(-4, 4, 9)[:, None]
    la, b = L.gates(alpha, -alpha, np.zeros(1), np.zeros(1))
    assert np.allclose(np.exp(la), 1.0 / (1.0 + np.exp(alpha)), rtol=1e-14)
    assert np.allclose(b, 1.0 / (1.0 + np.exp(alpha)), rtol=1e-14)
    # A_log = log 2 doubles the log-decay
    la2, _ = L.gates(alpha, alpha, np.full(1, math.log(2.0)), np.zeros(1))
    assert np.allclose(la2, 2 * la, rtol=1e-14)


def test_norms_closed_forms():
    c = np.full((1, 1, 16), 3.0)
    assert np.allclose(L.l2norm_heads(c, 0.0), 0.25)            # 3 / sqrt(16 * 9)
    rng = np.random.default_rng(0)
    x = rng.normal(size=(4, 3, 32))
    assert np.allclose(np.linalg.norm(L.l2norm_heads(x, 0.0), axis=-1), 1.0)
    o = rng.normal(size=(4, 2, 8))
    assert np.all(L.gated_rmsnorm(o, np.zeros_like(o), np.ones(8), 1e-6) == 0)  # SiLU(0) = 0
    oc = np.full((1, 1, 8), -2.0)
    r = L.gated_rmsnorm(oc, np.full_like(oc, 40.0), np.full(8, 0.5), 0.0)
    assert np.allclose(r, -1.0 * 0.5 * 40.0, rtol=1e-12)         # -2/2 * w * SiLU(40)
    assert np.array_equal(L.expand_kv_heads(np.arange(2)[None, :, None], 4)[0, :, 0], [0, 0, 1, 1])


# ----------------------------------------------------------------- conv

def test_conv_direct_sums():
    rng = np.random.default_rng(2)
    n, c = 6, 3
    x = rng.normal(size=(n, c))
    w = rng.normal(size=(c, 4))
    tail = rng.normal(size=(c, 3))
    u, new_tail = L.causal_conv(x, w, tail)
    hist = {ch: list(tail[ch]) + list(x[:, ch]) for ch in range(c)}   # x_{-3}, x_{-2}, x_{-1}, x_0, ...
    for t in range(n):
        for ch in range(c):
            ref = w[ch, 0] * hist[ch][t] + w[ch, 1] * hist[ch][t + 1] + w[ch, 2] * hist[ch][t + 2] + w[ch, 3] * hist[ch][t + 3]
            assert u[t, ch] == pytest.approx(ref, rel=1e-14, abs=1e-14)
    assert np.array_equal(new_tail, x[-3:].T)
    # fewer tokens than taps: the new tail mixes the old tail and the inputs
    u1, t1 = L.causal_conv(x[:1], w, tail)
    assert np.array_equal(t1, np.concatenate([tail[:, 1:], x[:1].T], axis=1))


def test_conv_split_equals_whole():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(11, 5))
    w = rng.normal(size=(5, 4))
    tail0 = np.zeros((5, 3))
    u, t = L.causal_conv(x, w, tail0)
    for cut in (1, 2, 3, 7):
        ua, ta = L.causal_conv(x[:cut], w, tail0)
        ub, tb = L.causal_conv(x[cut:], w, ta)
        assert np.array_equal(np.concatenate([ua, ub]), u)
        assert np.array_equal(tb, t)


# ----------------------------------------------------------------- recurrence

def _rand_case(rng, n, hv, dk, dv):
    q = rng.normal(size=(n, hv, dk))
    k = _unit(rng.normal(size=(n, hv, dk)))
    v = rng.normal(size=(n, hv, dv))
    la = -np.logaddexp(0, rng.normal(size=(n, hv)))
    b = 1 / (1 + np.exp(-rng.normal(size=(n, hv))))
    S0 = rng.normal(size=(hv, dv, dk))
    return q, k, v, la, b, S0


def check_recurrence_special_cases(rec):
    rng = np.random.default_rng(4)
    q, k, v, la, b, S0 = _rand_case(rng, 7, 2, 5, 3)
    # b = 0, a = 1: the state never changes and o_t = S_0 q_t
    o, S = rec(q, k, v, np.zeros_like(la), np.zeros_like(b), S0)
    assert np.allclose(S, S0, rtol=0, atol=1e-12)
    assert np.allclose(o, np.einsum("hij,thj->thi", S0, q), rtol=1e-12, atol=1e-12)
    # b = 0: pure decay, S_t = exp(sum log a) S_0
    o, S = rec(q, k, v, la, np.zeros_like(b), S0)
    assert np.allclose(S, np.exp(la.sum(0))[:, None, None] * S0, rtol=1e-12, atol=1e-14)
    # b = 1 with unit keys: the written key reads back its value, S_t k_t = v_t
    _, S1 = rec(q[:1], k[:1], v[:1], la[:1], np.ones_like(b[:1]), S0)
    assert np.allclose(np.einsum("hij,hj->hi", S1, k[0]), v[0], rtol=1e-12, atol=1e-12)
    # one token from the zero state: o = b (k . q) v
    o, _ = rec(q[:1], k[:1], v[:1], la[:1], b[:1], np.zeros_like(S0))
    ref = b[0][:, None] * np.einsum("hj,hj->h", k[0], q[0])[:, None] * v[0]
    assert np.allclose(o[0], ref, rtol=1e-12, atol=1e-14)


def check_recurrence_brute_force(rec):
    """S_N = S_0 P_1..P_N + sum_t b_t v_t k_t^T P_{t+1}..P_N with P_t = a_t (I - b_t k_t k_t^T),
    built from explicit matrices on tiny sizes; o_t = S_t q_t from the same products."""
    rng = np.random.default_rng(6)
    for n, dk, dv in [(1, 2, 2), (4, 3, 2), (6, 4, 4)]:
        q, k, v, la, b, S0 = _rand_case(rng, n, 1, dk, dv)
        k = rng.normal(size=k.shape)            # keys need not be unit here
        o, S = rec(q, k, v, la, b, S0)
        a = np.exp(la)
        P = [a[t, 0] * (np.eye(dk) - b[t, 0] * np.outer(k[t, 0], k[t, 0])) for t in range(n)]
        for upto in range(1, n + 1):
            St = S0[0].copy()
            for t in range(upto):
                St = St @ P[t]
            for t in range(upto):
                term = b[t, 0] * np.outer(v[t, 0], k[t, 0])
                for s in range(t + 1, upto):
                    term = term @ P[s]
                St = St + term
            assert np.allclose(o[upto - 1, 0], St @ q[upto - 1, 0], rtol=1e-10, atol=1e-12)
        assert np.allclose(S[0], St, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("check", [check_recurrence_special_cases, check_recurrence_brute_force])
def test_recurrence_pins_sequential(check):
    check(L.gated_delta_rule)


@pytest.mark.parametrize("chunk", [1, 3, 4, 64])
def test_recurrence_pins_chunked(chunk):
    rec = lambda *a: L.gated_delta_rule_chunked(*a, chunk=chunk)  # noqa: E731
    check_recurrence_special_cases(rec)
    check_recurrence_brute_force(rec)


def test_planted_missing_decay_is_caught():
    """Dropping a_t from the (S k) k^T term must fail the brute-force pin."""
    def wrong(q, k, v, log_a, b, S0):
        a = np.exp(log_a)
        S = np.array(S0, float)
        o = np.zeros(v.shape)
        for t in range(v.shape[0]):
            Sk = np.einsum("hij,hj->hi", S, k[t])[:, :, None]
            S = a[t][:, None, None] * S - b[t][:, None, None] * Sk * k[t][:, None, :] + b[t][:, None, None] * v[t][:, :, None] * k[t][:, None, :]
            o[t] = np.einsum("hij,hj->hi", S, q[t])
        return o, S
    with pytest.raises(AssertionError):
        check_recurrence_brute_force(wrong)


def test_planted_output_before_update_is_caught():
    """Reading o_t = S_{t-1} q_t (before the update) must fail the one-token pin."""
    def wrong(q, k, v, log_a, b, S0):
        a = np.exp(log_a)
        S = np.array(S0, float)
        o = np.zeros(v.shape)
        for t in range(v.shape[0]):
            o[t] = np.einsum("hij,hj->hi", S, q[t])
            Sk = np.einsum("hij,hj->hi", S, k[t])[:, :, None]
            S = a[t][:, None, None] * (S - b[t][:, None, None] * Sk * k[t][:, None, :]) + b[t][:, None, None] * v[t][:, :, None] * k[t][:, None, :]
        return o, S
    with pytest.raises(AssertionError):
        check_recurrence_special_cases(wrong)


@pytest.mark.parametrize("n,chunk", [(64, 64), (130, 64), (37, 16), (5, 64)])
def test_chunked_equals_sequential(n, chunk):
    rng = np.random.default_rng(n)
    q, k, v, la, b, S0 = _rand_case(rng, n, 3, 16, 8)
    q = _unit(q)
    o1, S1 = L.gated_delta_rule(q, k, v, la, b, S0)
    o2, S2 = L.gated_delta_rule_chunked(q, k, v, la, b, S0, chunk=chunk)
    assert np.linalg.norm(o1 - o2) <= 1e-10 * np.linalg.norm(o1)
    assert np.linalg.norm(S1 - S2) <= 1e-10 * np.linalg.norm(S1)


def test_planted_chunk_sign_error_is_caught(monkeypatch):
    """A chunked form with W added instead of subtracted must not match the sequential one."""
    rng = np.random.default_rng(9)
    q, k, v, la, b, S0 = _rand_case(rng, 20, 2, 8, 8)
    real_inv = np.linalg.inv
    monkeypatch.setattr(L.np.linalg, "inv", lambda m: real_inv(2 * np.eye(len(m)) - m))  # (I - Lm)^-1
    o2, S2 = L.gated_delta_rule_chunked(q, k, v, la, b, S0, chunk=8)
    monkeypatch.setattr(L.np.linalg, "inv", real_inv)
    o1, S1 = L.gated_delta_rule(q, k, v, la, b, S0)
    assert np.linalg.norm(o1 - o2) > 1e-3 * np.linalg.norm(o1)


@pytest.mark.parametrize("n,m", [(10, 7), (64, 65), (3, 1)])
def test_extend_equals_full(n, m):
    rng = np.random.default_rng(100 + n)
    q, k, v, la, b, S0 = _rand_case(rng, n + m, 2, 8, 8)
    o, S = L.gated_delta_rule(q, k, v, la, b, S0)
    oa, Sa = L.gated_delta_rule(q[:n], k[:n], v[:n], la[:n], b[:n], S0)
    ob, Sb = L.gated_delta_rule(q[n:], k[n:], v[n:], la[n:], b[n:], Sa)
    assert np.array_equal(np.concatenate([oa, ob]), o) and np.array_equal(Sb, S)
    oc, Sc = L.gated_delta_rule_chunked(q[:n], k[:n], v[:n], la[:n], b[:n], S0, chunk=16)
    od, Sd = L.gated_delta_rule_chunked(q[n:], k[n:], v[n:], la[n:], b[n:], Sc, chunk=16)
    assert np.linalg.norm(np.concatenate([oc, od]) - o) <= 1e-12 * np.linalg.norm(o)
    assert np.linalg.norm(Sd - S) <= 1e-12 * np.linalg.norm(S)


# ----------------------------------------------------------------- whole layer

def _params(spec, layer):
    p = dict(wtype=spec.wtype, hidden=spec.hidden, n_qk_heads=spec.n_qk_heads, n_v_heads=spec.n_v_heads,
             dk=spec.dk, dv=spec.dv, conv_w=layer["conv_w"], A_log=layer["A_log"], dt_bias=layer["dt_bias"],
             norm_w=layer["norm_w"], eps_l2=1e-6, eps_rms=1e-6, q_scale=spec.dk ** -0.5)
    if spec.wtype == "q4k":
        p["w_in"] = q4k.pack_q4k(layer["w_in"])
        p["w_out"] = q4k.pack_q4k(layer["w_out"])
    else:
        p["w_in"], p["w_out"] = layer["w_in"], layer["w_out"]
    return p


def _small_spec(wtype):
    return synth.LayerSpec("t", 256, 4, 8, 32, 32, 40, wtype, 0, "softplus_normal")


@pytest.mark.parametrize("wtype", ["q4k", "f32"])
def test_layer_extend_equals_full(wtype):
    spec = _small_spec(wtype)
    p = _params(spec, synth.make_layer(spec))
    tok = synth.make_tokens(spec, 40, seed=1)
    full = L.layer_forward(p, tok["x"], gate_log_a=tok["log_a"], gate_b=tok["b"])
    a = L.layer_forward(p, tok["x"][:25], gate_log_a=tok["log_a"][:25], gate_b=tok["b"][:25])
    b = L.layer_forward(p, tok["x"][25:], S0=a["state"], conv_tail=a["conv_tail"],
                        gate_log_a=tok["log_a"][25:], gate_b=tok["b"][25:])
    assert np.array_equal(np.concatenate([a["y"], b["y"]]), full["y"])
    assert np.array_equal(b["state"], full["state"])
    assert np.array_equal(b["conv_tail"], full["conv_tail"])


def test_layer_chunked_equals_sequential():
    spec = _small_spec("q4k")
    p = _params(spec, synth.make_layer(spec))
    tok = synth.make_tokens(spec, 40, seed=2)
    s = L.layer_forward(p, tok["x"], gate_log_a=tok["log_a"], gate_b=tok["b"])
    c = L.layer_forward(p, tok["x"], gate_log_a=tok["log_a"], gate_b=tok["b"], sequential=False, chunk=16)
    assert np.linalg.norm(s["o"] - c["o"]) <= 1e-10 * np.linalg.norm(s["o"])
    assert np.linalg.norm(s["y"] - c["y"]) <= 1e-2 * np.linalg.norm(s["y"])


def test_layer_projection_is_quantised_product():
    """The fused input projection of a Q4_K layer equals the int8 product of the decoded weights."""
    spec = _small_spec("q4k")
    layer = synth.make_layer(spec)
    p = _params(spec, layer)
    tok = synth.make_tokens(spec, 8, seed=3)
    qkvz, ba = L.project_in(p, tok["x"])
    # against the unquantised fp64 product: int8 rows carry ~1% relative error each
    ref = tok["x"].astype(np.float64) @ layer["w_in"].astype(np.float64).T
    got = np.concatenate([qkvz, ba], axis=1)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert 1e-3 < rel < 0.1
