"""Causal grouped-query attention for the prefill of the full-attention layers (oracle).

TEST INFRASTRUCTURE (see the package header).

The pages name flash attention for the hybrid model's full-attention layers as
the second prefill workload: "qwen35 batched prefill: flash attention for the
full-attention layers" (#5305, sub-ticket #4442), where the prefill rate falls
at 32k because those layers run "cuBLAS f32 with a materialised score matrix"
("CRUX parity spike" #4220, long-context finding 2), and the existing flash
path takes "f16 inputs, f32 accumulation".  The pages do not write the
operation out; the plain reading is standard causal softmax attention with
grouped key/value heads:

    for query head h (key/value head g = h // (Hq / Hkv)) and query i, at
    position p_i = nk - nq + i of the nk keys (the queries are the last nq
    positions, so nq = nk is a fresh prefill and nq < nk extends a held prefix):
        s_ij = scale * q_i . k_j          for j <= p_i
        o_i  = sum_j softmax_j(s_ij) v_j

computed here in float64 from the given (bf16-valued) inputs, one head at a
time, with the maximum subtracted before the exponential.
"""
from __future__ import annotations

import numpy as np


def attention(q, k, v, scale=None):
    """q [nq, Hq, D], k and v [nk, Hkv, D] -> o [nq, Hq, D] (float64)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    nq, hq, d = q.shape
    nk, hkv, _ = k.shape
    assert hq % hkv == 0 and nk >= nq
    if scale is None:
        scale = d ** -0.5
    pos = nk - nq + np.arange(nq)
    allowed = np.arange(nk)[None, :] <= pos[:, None]            # [nq, nk]
    o = np.empty((nq, hq, d))
    for h in range(hq):
        g = h // (hq // hkv)
        s = scale * (q[:, h, :] @ k[:, g, :].T)
        s = np.where(allowed, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        o[:, h, :] = p @ v[:, g, :]
    return o
