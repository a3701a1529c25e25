"""Pins for the oracle's whole-layer composition (projections, conv, gates,
delta rule, gated RMSNorm, output projection) on hand-built tiny layers.

The pages name the steps of one GDN layer and their order ("CRUX parity
spike" #4220, technique table row 2: projections, gates, conv, delta,
gated-norm; sparkinfer PR #464, Summary, "Token-parallel GDN conv": causal
4-tap conv over the raw inputs, SiLU, per-head L2 norm) but print no expected
output.  These tests write the expected values out by hand, element by
element, with Python's ``math`` module:

* fp32 layer: every row of W_in and W_out is a selector (one non-zero weight,
  a dyadic coefficient, at a permuted column), so every projection output is
  one input coordinate times a known coefficient, exact in bf16;
* Q4_K layer: the two quantised products are taken with the encoding
  primitives that ``test_oracle_quant.py`` and ``test_oracle_q4k.py`` pin
  (decode, int8 rows, exact integer product, fp32 rescale, bf16 rounding); the
  output projection quantises the whole token row of o_hat with one scale.

Everything between the two products follows the five steps directly: slices
q|k|v|z|beta|alpha of the fused projection, causal conv (tap 3 on the current
token), SiLU, L2 norm of each q/k head (q times q_scale afterwards), gates
log a = -exp(A_log) softplus(alpha + dt_bias) and b = sigmoid(beta), value
head h reading key head h // (Hv/Hk), the delta rule through explicit
transition matrices a_t (I - b_t k_t k_t^T) (one token from the zero state:
the closed form o = b (k.q) v), o / sqrt(mean o^2 + eps) * w * SiLU(z).

Each planted mistake below (beta and alpha swapped, q_scale on k, SiLU after
the norm, z read from the wrong slice, o_hat quantised per head, the key-head
map h mod Hk, the conv taps reversed) must fail a pin.
"""
import math

import numpy as np
import pytest

from oracle import layer as L
from oracle import q4k
from oracle import quant

# --------------------------------------------------------------- scalar math


def _silu(u):
    return u / (1.0 + math.exp(-u))


def _sigmoid(u):
    return 1.0 / (1.0 + math.exp(-u))


def _softplus(u):
    return math.log(1.0 + math.exp(u))


# --------------------------------------------------------------- the layers

HK, HV, DK, DV = 2, 4, 2, 2            # fp32 selector layer: 2 key heads, 4 value heads (2:1)
C_QK, C_V = HK * DK, HV * DV
C_CONV = 2 * C_QK + C_V
R_IN = 2 * C_QK + 2 * C_V + 2 * HV     # q | k | v | z | beta | alpha = 32 rows
H_SEL = 32


def _perm(r, n):
    return (5 * r + 3) % n             # a permutation of 0..n-1 (gcd(5, n) = 1 for n = 32)


def _selector_layer(taps):
    """fp32 layer whose W_in row r holds c_r at column perm(r) and W_out row j holds
    d_j at column (3 j + 1) mod C_v; c_r, d_j are dyadic with at most 3 significant bits."""
    c = np.array([(0.5, 0.625, 0.75, 1.25)[r % 4] * (-1.0 if r % 3 == 1 else 1.0) for r in range(R_IN)])
    w_in = np.zeros((R_IN, H_SEL), np.float32)
    for r in range(R_IN):
        w_in[r, _perm(r, H_SEL)] = c[r]
    d = np.array([(1.0, -0.75, 0.5, 1.5)[j % 4] for j in range(H_SEL)])
    w_out = np.zeros((H_SEL, C_V), np.float32)
    for j in range(H_SEL):
        w_out[j, (3 * j + 1) % C_V] = d[j]
    if taps == "current":
        conv_w = np.zeros((C_CONV, 4))
        conv_w[:, 3] = 1.0
    else:                               # a known pattern, different per channel
        conv_w = np.array([[0.25 + 0.01 * ch, -0.5, 0.125 * (1 + ch % 3), 1.0 - 0.02 * ch] for ch in range(C_CONV)])
    p = dict(wtype="f32", hidden=H_SEL, n_qk_heads=HK, n_v_heads=HV, dk=DK, dv=DV, w_in=w_in, w_out=w_out,
             conv_w=conv_w, A_log=np.array([0.3, -0.2, 0.1, 0.5]), dt_bias=np.array([0.1, -0.4, 0.25, 0.0]),
             norm_w=np.array([1.1, 0.9]), eps_l2=0.05, eps_rms=0.03, q_scale=0.7)
    return p, c, d


def _selector_tokens(n, seed):
    """x[t, j] = (2 m - 31) / 16 for a seeded permutation m of 0..31: distinct, 5 significant bits."""
    rng = np.random.default_rng(seed)
    return np.stack([(2.0 * rng.permutation(H_SEL) - 31.0) / 16.0 for _ in range(n)]).astype(np.float32)


# --------------------------------------------------------------- closed form

def _expected(p, P, S0, tail, out_proj):
    """The five steps by hand, from the fused projection rows P[t][r] (a list per token).

    S0: nested lists [Hv][dv][dk] or None (zero state); tail: [C_conv][3] or None.
    out_proj(o_hat_row) -> y row.  Returns dict of y, state, o, o_hat, conv_tail."""
    hk, hv, dk, dv = p["n_qk_heads"], p["n_v_heads"], p["dk"], p["dv"]
    c_qk, c_v = hk * dk, hv * dv
    c_conv = 2 * c_qk + c_v
    n = len(P)
    zero_state = S0 is None
    S = [[[0.0] * dk for _ in range(dv)] for _ in range(hv)] if zero_state else [[list(r) for r in m] for m in S0]
    hist = [[0.0, 0.0, 0.0] if tail is None else list(tail[ch]) for ch in range(c_conv)]
    W = p["conv_w"]
    out = {"y": [], "o": [], "o_hat": []}
    for t in range(n):
        row = P[t]
        for ch in range(c_conv):
            hist[ch].append(float(row[ch]))
        # step 2: causal conv (x_{t-3} .. x_t against taps 0..3), SiLU
        act = [_silu(sum(W[ch][j] * hist[ch][t + j] for j in range(4))) for ch in range(c_conv)]
        qh, kh = [], []
        for g in range(hk):
            qa = act[g * dk:(g + 1) * dk]
            ka = act[c_qk + g * dk:c_qk + (g + 1) * dk]
            nq = math.sqrt(sum(e * e for e in qa) + p["eps_l2"])
            nk = math.sqrt(sum(e * e for e in ka) + p["eps_l2"])
            qh.append([p["q_scale"] * e / nq for e in qa])
            kh.append([e / nk for e in ka])
        ohat_row = []
        o_t = []
        for h in range(hv):
            g = h // (hv // hk)
            q, k = qh[g], kh[g]
            v = act[2 * c_qk + h * dv:2 * c_qk + (h + 1) * dv]
            z = row[c_conv + h * dv:c_conv + (h + 1) * dv]
            beta = row[c_conv + c_v + h]
            alpha = row[c_conv + c_v + hv + h]
            b = _sigmoid(beta)
            a = math.exp(-math.exp(p["A_log"][h]) * _softplus(alpha + p["dt_bias"][h]))
            if zero_state and t == 0:
                # one token from the zero state: S_1 = b v k^T, o = b (k . q) v
                kq = sum(k[j] * q[j] for j in range(dk))
                o = [b * kq * v[i] for i in range(dv)]
                S[h] = [[b * v[i] * k[j] for j in range(dk)] for i in range(dv)]
            elif dk <= 8:
                # S_t = S_{t-1} P_t + b v k^T with the transition matrix P_t = a (I - b k k^T)
                Pm = [[a * ((1.0 if i == j else 0.0) - b * k[i] * k[j]) for j in range(dk)] for i in range(dk)]
                S[h] = [[sum(S[h][i][m] * Pm[m][j] for m in range(dk)) + b * v[i] * k[j] for j in range(dk)]
                        for i in range(dv)]
                o = [sum(S[h][i][j] * q[j] for j in range(dk)) for i in range(dv)]
            else:
                # the same product row by row: row i of S_{t-1} P_t is a (s_i - b (s_i . k) k)
                for i in range(dv):
                    si = S[h][i]
                    sk = sum(si[m] * k[m] for m in range(dk))
                    S[h][i] = [a * (si[j] - b * sk * k[j]) + b * v[i] * k[j] for j in range(dk)]
                o = [sum(S[h][i][j] * q[j] for j in range(dk)) for i in range(dv)]
            o_t.append(o)
            # step 4: gated RMSNorm
            rms = math.sqrt(sum(e * e for e in o) / dv + p["eps_rms"])
            ohat_row += [o[i] / rms * p["norm_w"][i] * _silu(float(z[i])) for i in range(dv)]
        out["o"].append(o_t)
        out["o_hat"].append(ohat_row)
        out["y"].append(out_proj(ohat_row))
    out["state"] = S
    out["conv_tail"] = [hist[ch][-3:] for ch in range(c_conv)]
    return {k_: np.array(v_, np.float64) for k_, v_ in out.items()}


def _given_state(hv, dv, dk, seed):
    rng = np.random.default_rng(seed)
    return rng.normal(scale=0.5, size=(hv, dv, dk)), rng.normal(size=(2 * HK * DK + HV * DV, 3))


def _rel(a, b):
    return np.linalg.norm(np.asarray(a, np.float64) - np.asarray(b, np.float64)) / np.linalg.norm(b)


def check_selector_layer(n, given, taps):
    p, c, d = _selector_layer(taps)
    x = _selector_tokens(n, seed=10 * n + (1 if given else 0))
    S0, tail = (None, None)
    if given:
        S0, tail = _given_state(HV, DV, DK, seed=n)
    # the selector product: row r of the fused projection is c_r * x[perm(r)]
    P = [[c[r] * float(x[t][_perm(r, H_SEL)]) for r in range(R_IN)] for t in range(n)]
    out_proj = lambda oh: [d[j] * oh[(3 * j + 1) % C_V] for j in range(H_SEL)]  # noqa: E731
    exp = _expected(p, P, None if S0 is None else S0.tolist(), None if tail is None else tail.tolist(), out_proj)
    got = L.layer_forward(p, x, S0=S0, conv_tail=tail)
    assert _rel(got["o"], exp["o"]) <= 1e-12
    assert _rel(got["state"], exp["state"]) <= 1e-12
    assert _rel(got["o_hat"].reshape(n, C_V), exp["o_hat"]) <= 1e-12
    assert _rel(got["y"], exp["y"]) <= 1e-6            # y is float32 for an fp32 layer
    assert np.array_equal(np.asarray(got["conv_tail"], np.float64), exp["conv_tail"])


CASES = [(1, False, "current"), (2, False, "current"), (1, True, "current"), (2, True, "current"),
         (1, False, "pattern"), (2, True, "pattern"), (5, True, "pattern")]


@pytest.mark.parametrize("n,given,taps", CASES)
def test_selector_layer_closed_form(n, given, taps):
    check_selector_layer(n, given, taps)


def test_selector_layer_one_token_values():
    """Spot values of the one-token, zero-state, current-tap case, from the closed
    form o = b (k.q) v with the gates of the layer fields (no override)."""
    p, c, d = _selector_layer("current")
    x = _selector_tokens(1, seed=10)
    got = L.layer_forward(p, x)
    P = [c[r] * float(x[0][_perm(r, H_SEL)]) for r in range(R_IN)]
    # value head 3 reads key head 1; beta_3 = P[24 + 3], alpha_3 = P[28 + 3]
    b3 = 1.0 / (1.0 + math.exp(-P[27]))
    qa = [_silu(P[2]), _silu(P[3])]
    ka = [_silu(P[6]), _silu(P[7])]
    qn = [0.7 * e / math.sqrt(qa[0] ** 2 + qa[1] ** 2 + 0.05) for e in qa]
    kn = [e / math.sqrt(ka[0] ** 2 + ka[1] ** 2 + 0.05) for e in ka]
    v3 = [_silu(P[8 + 6]), _silu(P[8 + 7])]
    o3 = [b3 * (qn[0] * kn[0] + qn[1] * kn[1]) * e for e in v3]
    assert got["o"][0, 3] == pytest.approx(o3, rel=1e-13)
    assert got["b"][0, 3] == pytest.approx(b3, rel=1e-15)
    la3 = -math.exp(0.5) * math.log1p(math.exp(P[31] + 0.0))
    assert got["log_a"][0, 3] == pytest.approx(la3, rel=1e-13)


# --------------------------------------------------------------- Q4_K layer

QH, QHK, QHV, QD = 256, 1, 2, 128      # hidden 256, 1 key head, 2 value heads of 128


def _q4k_layer(seed):
    rng = np.random.default_rng(seed)
    r_in = 2 * QHK * QD + 2 * QHV * QD + 2 * QHV
    w_in = rng.normal(scale=0.02, size=(r_in, QH)).astype(np.float32)
    # make the two value heads' outputs differ in scale, so per-row and per-head quantisation differ
    w_in[2 * QD + QD:2 * QD + 2 * QD] *= 4.0
    w_out = rng.normal(scale=0.02, size=(QH, QHV * QD)).astype(np.float32)
    c_conv = 2 * QHK * QD + QHV * QD
    p = dict(wtype="q4k", hidden=QH, n_qk_heads=QHK, n_v_heads=QHV, dk=QD, dv=QD,
             w_in=q4k.pack_q4k(w_in), w_out=q4k.pack_q4k(w_out),
             conv_w=rng.normal(scale=0.3, size=(c_conv, 4)), A_log=np.array([0.2, -0.3]),
             dt_bias=np.array([0.5, -0.1]), norm_w=1.0 + rng.normal(scale=0.1, size=QD),
             eps_l2=1e-6, eps_rms=1e-6, q_scale=QD ** -0.5)
    return p


def check_q4k_layer(n, given):
    p = _q4k_layer(7)
    rng = np.random.default_rng(20 + n)
    x = quant.bf16_round(rng.normal(size=(n, QH)).astype(np.float32))
    c_conv = 2 * QHK * QD + QHV * QD
    S0 = rng.normal(scale=0.3, size=(QHV, QD, QD)) if given else None
    tail = rng.normal(size=(c_conv, 3)) if given else None
    r_in = 2 * QHK * QD + 2 * QHV * QD + 2 * QHV
    # step 1 with the pinned encodings: int8 rows of x and of the decoded W_in, exact product,
    # fp32 rescale; q|k|v|z rounded to bf16, beta|alpha kept in fp32
    qx, sx = quant.quant_rows_i8(x)
    qw, sw = quant.quant_rows_i8(q4k.unpack_q4k(p["w_in"], r_in, QH))
    P = quant.gemm_q8(qx, sx, qw, sw)
    nb = 2 * QHK * QD + 2 * QHV * QD
    P = np.concatenate([quant.bf16_round(P[:, :nb]), P[:, nb:]], axis=1).astype(np.float64)
    qo_w, so_w = quant.quant_rows_i8(q4k.unpack_q4k(p["w_out"], QH, QHV * QD))

    def out_proj(oh):                   # step 5: one int8 scale for the whole token row
        qo, so = quant.quant_rows_i8(np.array([oh], np.float32))
        return quant.bf16_round(quant.gemm_q8(qo, so, qo_w, so_w))[0].astype(np.float64).tolist()

    exp = _expected(p, P.tolist(), None if S0 is None else S0.tolist(), None if tail is None else tail.tolist(),
                    out_proj)
    got = L.layer_forward(p, x, S0=S0, conv_tail=tail)
    assert _rel(got["o"], exp["o"]) <= 1e-12
    assert _rel(got["state"], exp["state"]) <= 1e-12
    assert _rel(got["o_hat"].reshape(n, -1), exp["o_hat"]) <= 1e-12
    assert _rel(got["y"], exp["y"]) <= 1e-6


@pytest.mark.parametrize("n,given", [(1, False), (2, True)])
def test_q4k_layer_closed_form(n, given):
    check_q4k_layer(n, given)


# --------------------------------------------------------------- planted mistakes

def _wrong_conv_stage(q_scale_on_k=False, silu_after_norm=False):
    def conv_stage(p, qkv_raw, tail):
        sz = L.layer_sizes(p)
        n = qkv_raw.shape[0]
        u, new_tail = L.causal_conv(qkv_raw, p["conv_w"], tail)
        c_qk = sz["c_qk"]
        if silu_after_norm:
            y = u
            q = L.silu(L.l2norm_heads(y[:, :c_qk].reshape(n, p["n_qk_heads"], p["dk"]), p["eps_l2"]))
            k = L.silu(L.l2norm_heads(y[:, c_qk:2 * c_qk].reshape(n, p["n_qk_heads"], p["dk"]), p["eps_l2"]))
            q = q * p["q_scale"]
            v = L.silu(y[:, 2 * c_qk:]).reshape(n, p["n_v_heads"], p["dv"])
        else:
            y = L.silu(u)
            q = L.l2norm_heads(y[:, :c_qk].reshape(n, p["n_qk_heads"], p["dk"]), p["eps_l2"])
            k = L.l2norm_heads(y[:, c_qk:2 * c_qk].reshape(n, p["n_qk_heads"], p["dk"]), p["eps_l2"])
            if q_scale_on_k:
                k = k * p["q_scale"]
            else:
                q = q * p["q_scale"]
            v = y[:, 2 * c_qk:].reshape(n, p["n_v_heads"], p["dv"])
        return q, k, v, new_tail
    return conv_stage


def _check_all():
    for n, given, taps in CASES:
        check_selector_layer(n, given, taps)
    check_q4k_layer(1, False)
    check_q4k_layer(2, True)


def test_planted_beta_alpha_swap_is_caught(monkeypatch):
    real = L.gates
    monkeypatch.setattr(L, "gates", lambda alpha, beta, A_log, dt_bias: real(beta, alpha, A_log, dt_bias))
    with pytest.raises(AssertionError):
        _check_all()


def test_planted_q_scale_on_k_is_caught(monkeypatch):
    monkeypatch.setattr(L, "conv_stage", _wrong_conv_stage(q_scale_on_k=True))
    with pytest.raises(AssertionError):
        _check_all()


def test_planted_silu_after_norm_is_caught(monkeypatch):
    monkeypatch.setattr(L, "conv_stage", _wrong_conv_stage(silu_after_norm=True))
    with pytest.raises(AssertionError):
        _check_all()


def test_planted_wrong_z_slice_is_caught(monkeypatch):
    """z read from the v slice of the fused projection instead of its own."""
    real = L.project_in

    def project_in(p, x32, decode=False):
        qkvz, ba = real(p, x32, decode=decode)
        sz = L.layer_sizes(p)
        qkvz = qkvz.copy()
        qkvz[:, sz["c_conv"]:] = qkvz[:, 2 * sz["c_qk"]:2 * sz["c_qk"] + sz["c_v"]]
        return qkvz, ba
    monkeypatch.setattr(L, "project_in", project_in)
    with pytest.raises(AssertionError):
        _check_all()


def test_planted_per_head_output_quantisation_is_caught(monkeypatch):
    real = L.project_out

    def project_out(p, o_hat, decode=False):
        if p["wtype"] != "q4k":
            return real(p, o_hat, decode=decode)
        sz = L.layer_sizes(p)
        wf = L.unpack_weights(p, "w_out", p["hidden"], sz["c_v"])
        qw, sw = quant.quant_rows_i8(wf)
        oh = np.asarray(o_hat, np.float64).astype(np.float32)
        acc = np.zeros((oh.shape[0], p["hidden"]), np.float32)
        for h in range(p["n_v_heads"]):
            sl = slice(h * p["dv"], (h + 1) * p["dv"])
            qo, so = quant.quant_rows_i8(oh[:, sl])
            acc += quant.rescale(quant.int_matmul_exact(qo, qw[:, sl]), so, sw)
        return quant.bf16_round(acc)
    monkeypatch.setattr(L, "project_out", project_out)
    with pytest.raises(AssertionError):
        check_q4k_layer(1, False)


def test_planted_key_head_modulo_map_is_caught(monkeypatch):
    monkeypatch.setattr(L, "expand_kv_heads", lambda x, hv: np.tile(x, (1, hv // x.shape[1], 1)))
    with pytest.raises(AssertionError):
        _check_all()


def test_planted_reversed_conv_taps_is_caught(monkeypatch):
    real = L.causal_conv
    monkeypatch.setattr(L, "causal_conv", lambda x, w, tail: real(x, np.asarray(w)[:, ::-1], tail))
    with pytest.raises(AssertionError):
        _check_all()
