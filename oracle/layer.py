"""One Gated DeltaNet (GDN) layer, batched prefill, in fp64 (oracle).

TEST INFRASTRUCTURE (see the package header).

The pages list the steps of one GDN layer but not their formulas:

* "CRUX parity spike: apr serve vs ollama on Qwen3.5" (technique table, row
  2) names the per-layer kernels: projections, gates, conv, delta, gated-norm.
* sparkinfer PR #464 (Summary, "Token-parallel GDN conv"): a causal 4-tap conv
  over the raw inputs, then SiLU and a per-head L2 norm; the prompt starts at
  position 0, and a conv state carries the raw inputs across calls.
* "Verbs Are Fast" epic #3598 (parked tickets): the delta rule in a
  chunk-resident scan or the "WY-chunked (tensor-core) form".
* "Qwen3.5 on CPU prefills one token at a time" #5475 (What we already know):
  the DeltaNet recurrence runs per head; a prompt that extends the held tokens
  prefills only the suffix from the held state.

The recurrence is the gated delta rule of Gated DeltaNet (Yang, Kautz and
Hatamizadeh, "Gated Delta Networks", 2024), per value head, with the state
S (dv x dk) updated after each token:

    S_t = a_t * S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,     o_t = S_t q_t

Readings where the pages are silent (all are also stated in the design notes):
conv over the q|k|v channels only, tap 3 on the current token, the conv state
holding the last 3 raw inputs per channel oldest first; L2 norm
x / sqrt(sum x^2 + eps); q scaled by q_scale after its norm; value head h reads
key head floor(h / (Hv/Hk)); log a = -exp(A_log) * softplus(alpha + dt_bias)
and b = sigmoid(beta) unless drawn directly; gated RMSNorm
o / sqrt(mean o^2 + eps) * w * SiLU(z).
"""
from __future__ import annotations

import numpy as np

from . import q4k as _q4k
from . import q6k as _q6k
from . import quant as _quant

f64 = np.float64


# ---------------------------------------------------------------- elementwise

def silu(u):
    u = np.asarray(u, f64)
    return u / (1.0 + np.exp(-u))


def sigmoid(u):
    u = np.asarray(u, f64)
    return 1.0 / (1.0 + np.exp(-u))


def softplus(u):
    u = np.asarray(u, f64)
    return np.maximum(u, 0.0) + np.log1p(np.exp(-np.abs(u)))


# ---------------------------------------------------------------- conv + norms

def causal_conv(x_raw, conv_w, tail):
    """Causal depthwise conv, 4 taps (sparkinfer PR #464, "Token-parallel GDN conv").

    x_raw [N, C], conv_w [C, 4] (tap 3 multiplies the current token),
    tail [C, 3] = the 3 raw inputs before x_raw[0], oldest first.
    Returns u [N, C] with u_t = sum_j conv_w[:, j] * x_{t-3+j}, and the new tail."""
    x_raw = np.asarray(x_raw, f64)
    n = x_raw.shape[0]
    taps = conv_w.shape[1]
    ext = np.concatenate([np.asarray(tail, f64).T, x_raw], axis=0)  # ext[i] = x_{i-3}
    u = np.zeros_like(x_raw)
    for j in range(taps):
        u += np.asarray(conv_w, f64)[:, j][None, :] * ext[j:j + n]
    return u, ext[-(taps - 1):].T.copy()


def l2norm_heads(x, eps):
    """x [..., d] / sqrt(sum x^2 + eps) over the last axis (per head)."""
    x = np.asarray(x, f64)
    return x / np.sqrt((x * x).sum(axis=-1, keepdims=True) + eps)


def gates(alpha, beta, A_log, dt_bias):
    """log a = -exp(A_log) * softplus(alpha + dt_bias), b = sigmoid(beta); [N, Hv]."""
    log_a = -np.exp(np.asarray(A_log, f64))[None, :] * softplus(np.asarray(alpha, f64) + np.asarray(dt_bias, f64)[None, :])
    return log_a, sigmoid(beta)


def gated_rmsnorm(o, z, w, eps):
    """o, z [N, Hv, dv]: o / sqrt(mean(o^2) + eps) * w * SiLU(z), per head."""
    o = np.asarray(o, f64)
    r = o / np.sqrt((o * o).mean(axis=-1, keepdims=True) + eps)
    return r * np.asarray(w, f64)[None, None, :] * silu(z)


def expand_kv_heads(x, n_v_heads):
    """[N, Hk, d] -> [N, Hv, d]: value head h reads key head floor(h / (Hv/Hk))."""
    r = n_v_heads // x.shape[1]
    return np.repeat(x, r, axis=1)


# ---------------------------------------------------------------- recurrence

def gated_delta_rule(q, k, v, log_a, b, S0):
    """Sequential gated delta rule, one token at a time, fp64.

    q, k [N, Hv, dk]; v [N, Hv, dv]; log_a, b [N, Hv]; S0 [Hv, dv, dk].
    Returns o [N, Hv, dv] (o_t = S_t q_t, after the update) and S_N."""
    q, k, v = (np.asarray(t, f64) for t in (q, k, v))
    a = np.exp(np.asarray(log_a, f64))
    b = np.asarray(b, f64)
    S = np.array(S0, f64, copy=True)
    n, hv, dv = v.shape
    o = np.zeros((n, hv, dv), f64)
    for t in range(n):
        kt = k[t][:, None, :]                        # [Hv, 1, dk]
        Sk = np.einsum("hij,hj->hi", S, k[t])[:, :, None]
        S = a[t][:, None, None] * (S - b[t][:, None, None] * Sk * kt) + b[t][:, None, None] * v[t][:, :, None] * kt
        o[t] = np.einsum("hij,hj->hi", S, q[t])
    return o, S


def gated_delta_rule_chunked(q, k, v, log_a, b, S0, chunk=64):
    """The same recurrence in chunked WY/UT form, fp64 ("WY-chunked (tensor-core) form").

    Within a chunk (tokens 1..L, state S entering it), with gamma_i = sum_{j<=i} log a_j:
        Lm_ij = b_i e^{gamma_i - gamma_j} k_i.k_j  (j < i),   T = (I + Lm)^{-1}
        W = T diag(b e^gamma) K,   U = T diag(b) V,   Delta = U - W S^T
        O = diag(e^gamma) Q S^T + (M o Q K^T) Delta,   M_ij = e^{gamma_i - gamma_j} (j <= i)
        S <- e^{gamma_L} S + Delta^T diag(e^{gamma_L - gamma}) K
    """
    q, k, v = (np.asarray(t, f64) for t in (q, k, v))
    log_a = np.asarray(log_a, f64)
    b = np.asarray(b, f64)
    S = np.array(S0, f64, copy=True)
    n, hv, dv = v.shape
    o = np.zeros((n, hv, dv), f64)
    for c0 in range(0, n, chunk):
        c1 = min(n, c0 + chunk)
        L = c1 - c0
        g = np.cumsum(log_a[c0:c1], axis=0)          # [L, Hv]
        tri_strict = np.tril(np.ones((L, L)), -1)
        tri_incl = np.tril(np.ones((L, L)))
        for h in range(hv):
            K = k[c0:c1, h]
            Q = q[c0:c1, h]
            V = v[c0:c1, h]
            bh = b[c0:c1, h]
            gh = g[:, h]
            decay = np.exp(gh[:, None] - gh[None, :])
            Lm = tri_strict * (bh[:, None] * decay * (K @ K.T))
            T = np.linalg.inv(np.eye(L) + Lm)
            W = T @ ((bh * np.exp(gh))[:, None] * K)
            U = T @ (bh[:, None] * V)
            delta = U - W @ S[h].T
            O = np.exp(gh)[:, None] * (Q @ S[h].T) + (tri_incl * decay * (Q @ K.T)) @ delta
            o[c0:c1, h] = O
            S[h] = np.exp(gh[-1]) * S[h] + delta.T @ (np.exp(gh[-1] - gh)[:, None] * K)
    return o, S


# ---------------------------------------------------------------- whole layer

def layer_sizes(p):
    hk, hv, dk, dv = p["n_qk_heads"], p["n_v_heads"], p["dk"], p["dv"]
    c_qk, c_v = hk * dk, hv * dv
    return {"c_qk": c_qk, "c_v": c_v, "c_conv": 2 * c_qk + c_v, "n_bf16": 2 * c_qk + 2 * c_v,
            "r_in": 2 * c_qk + 2 * c_v + 2 * hv}


def unpack_weights(p, name, rows, cols):
    """Decode a quantised weight matrix: Q4_K, or Q6_K when p[name + "_fmt"] is
    "q6k" (the pages' fused dequant takes both formats: sparkinfer PR #464,
    Summary, "Fused Q4_K/Q6_K -> int8-row dequant")."""
    if p.get(name + "_fmt", "q4k") == "q6k":
        return _q6k.unpack_q6k(p[name], rows, cols)
    return _q4k.unpack_q4k(p[name], rows, cols)


def project_in(p, x32, decode=False):
    """Fused input projection P = x W_in^T split into bf16 q|k|v|z and fp32 beta|alpha.

    Q4_K layers: both operands int8 row-quantised, exact integer product, fp32
    rescale (sparkinfer PR #464, Summary).  decode: the decode step's product
    of the int8 activation rows with the exactly decoded weights
    (quant.matvec_exact_weights), rounded once to fp32.  fp32 layers: plain
    product."""
    sz = layer_sizes(p)
    if p["wtype"] == "q4k":
        wf = unpack_weights(p, "w_in", sz["r_in"], p["hidden"])
        qx, sx = _quant.quant_rows_i8(x32)
        if decode:
            P = _quant.matvec_exact_weights(qx, sx, wf).astype(np.float32)
        else:
            qw, sw = _quant.quant_rows_i8(wf)
            P = _quant.gemm_q8(qx, sx, qw, sw)
    else:
        P = (np.asarray(x32, f64) @ np.asarray(p["w_in"], f64).T).astype(np.float32)
    nb = sz["n_bf16"]
    return _quant.bf16_round(P[:, :nb]), P[:, nb:].copy()


def project_out(p, o_hat, decode=False):
    """Output projection y = o_hat W_out^T; Q4_K layers quantise o_hat (fp32) per
    token row (decode: against the exactly decoded weights, as project_in)."""
    sz = layer_sizes(p)
    if p["wtype"] == "q4k":
        wf = unpack_weights(p, "w_out", p["hidden"], sz["c_v"])
        qo, so = _quant.quant_rows_i8(np.asarray(o_hat, f64).astype(np.float32))
        if decode:
            return _quant.bf16_round(_quant.matvec_exact_weights(qo, so, wf).astype(np.float32))
        qw, sw = _quant.quant_rows_i8(wf)
        return _quant.bf16_round(_quant.gemm_q8(qo, so, qw, sw))
    return (np.asarray(o_hat, f64) @ np.asarray(p["w_out"], f64).T).astype(np.float32)


def conv_stage(p, qkv_raw, tail):
    """Conv + SiLU + per-head L2 norm (q, k) + q scale; returns q, k [N, Hk, dk], v [N, Hv, dv], new tail."""
    sz = layer_sizes(p)
    n = qkv_raw.shape[0]
    u, new_tail = causal_conv(qkv_raw, p["conv_w"], tail)
    y = silu(u)
    c_qk = sz["c_qk"]
    q = l2norm_heads(y[:, :c_qk].reshape(n, p["n_qk_heads"], p["dk"]), p["eps_l2"]) * p["q_scale"]
    k = l2norm_heads(y[:, c_qk:2 * c_qk].reshape(n, p["n_qk_heads"], p["dk"]), p["eps_l2"])
    v = y[:, 2 * c_qk:].reshape(n, p["n_v_heads"], p["dv"])
    return q, k, v, new_tail


def layer_forward(p, x32, S0=None, conv_tail=None, gate_log_a=None, gate_b=None, sequential=True, chunk=64,
                  decode=False):
    """Whole layer: projections, conv, gates, gated delta rule, gated RMSNorm, output projection.

    x32 [N, hidden] float32 (the exact values of the bf16 input for Q4_K layers);
    S0 [Hv, dv, dk] or None (zero state); conv_tail [C_conv, 3] or None (zeros).
    Returns a dict of every intermediate (float64 unless an encoding fixes it)."""
    sz = layer_sizes(p)
    n = x32.shape[0]
    hv, dv, dk = p["n_v_heads"], p["dv"], p["dk"]
    if S0 is None:
        S0 = np.zeros((hv, dv, dk))
    if conv_tail is None:
        conv_tail = np.zeros((sz["c_conv"], p["conv_w"].shape[1] - 1))
    qkvz, ba = project_in(p, x32, decode=decode)
    q, k, v, new_tail = conv_stage(p, qkvz[:, :sz["c_conv"]], conv_tail)
    z = qkvz[:, sz["c_conv"]:].reshape(n, hv, dv)
    if gate_log_a is not None:
        log_a, b = np.asarray(gate_log_a, f64), np.asarray(gate_b, f64)
    else:
        log_a, b = gates(ba[:, hv:2 * hv], ba[:, :hv], p["A_log"], p["dt_bias"])
    qe, ke = expand_kv_heads(q, hv), expand_kv_heads(k, hv)
    rec = gated_delta_rule if sequential else (lambda *a: gated_delta_rule_chunked(*a, chunk=chunk))
    o, S = rec(qe, ke, v, log_a, b, S0)
    o_hat = gated_rmsnorm(o, z, p["norm_w"], p["eps_rms"])
    y = project_out(p, o_hat.reshape(n, sz["c_v"]), decode=decode)
    return {"qkvz": qkvz, "ba": ba, "q": q, "k": k, "v": v, "z": z, "log_a": log_a, "b": b,
            "o": o, "state": S, "o_hat": o_hat, "y": y, "conv_tail": new_tail}
