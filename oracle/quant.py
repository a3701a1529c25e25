"""int8 row quantisation, the exact int8 x int8 product and bf16 rounding (oracle).

TEST INFRASTRUCTURE (see the package header).

sparkinfer PR #464 ("fused Q4K/Q6K->int8 dequant + token-parallel GDN conv
..."), Summary: the fused dequant writes "int8 + per-row scale directly", and
(Correctness paragraph) "quantizes from the exact fp32 dequant instead of the
bf16-rounded scratch".  The same page's int8 tensor-core GEMM consumes those
rows.  The pages fix neither the scale nor the rounding; the plain reading,
taken on both sides, is symmetric per-row quantisation in fp32:

    s = amax / 127                (IEEE fp32 divide)
    q = clamp(rne(w / s), -127, 127)   (IEEE fp32 divide, nearest-even)
    amax == 0  ->  s = 0, q = 0

and the product of two such matrices is the exact integer sum, rescaled in
fp32 as ((float)acc * s_row) * s_col, each step rounded to nearest-even.
"""
from __future__ import annotations

import numpy as np


def quant_rows_i8(w: np.ndarray):
    """Per-row symmetric int8 quantisation of float32 [R, K] -> (int8 [R, K], float32 [R])."""
    w = np.ascontiguousarray(w, np.float32)
    amax = np.abs(w).max(axis=-1)
    s = (amax / np.float32(127)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (w / np.where(s > 0, s, np.float32(1))[..., None]).astype(np.float32)
    q = np.clip(np.rint(r), -127, 127)
    q = np.where(s[..., None] > 0, q, 0).astype(np.int8)
    return q, s


def int_matmul_exact(qa: np.ndarray, qb: np.ndarray) -> np.ndarray:
    """Exact integer qa [M, K] @ qb [N, K]^T as int64.

    Carried out as a float64 matmul: every product and every partial sum is an
    integer below 127*127*K < 2^53 for K < 2^38, so float64 holds each one
    exactly whatever the summation order."""
    acc = qa.astype(np.float64) @ qb.astype(np.float64).T
    return acc.astype(np.int64)


def rescale(acc: np.ndarray, sa: np.ndarray, sb: np.ndarray) -> np.ndarray:
    """fp32 epilogue ((float)acc * sa[m]) * sb[n]; int64 -> float32 rounds to nearest-even."""
    y = acc.astype(np.float32) * sa.astype(np.float32)[:, None]
    return (y.astype(np.float32) * sb.astype(np.float32)[None, :]).astype(np.float32)


def gemm_q8(qa, sa, qb, sb) -> np.ndarray:
    """Quantised projection: rescaled exact integer product, float32 [M, N]."""
    return rescale(int_matmul_exact(qa, qb), sa, sb)


def matvec_exact_weights(qa: np.ndarray, sa: np.ndarray, w: np.ndarray) -> np.ndarray:
    """The decode step's projection: int8 row codes qa [M, K] with scales sa [M]
    against the exactly decoded weights w [N, K] (no re-quantisation of the
    weights), y = sa[m] * sum_k qa[m, k] w[n, k], in float64.

    This is the quantised-activation product of a decode GEMV that reads the
    4-bit or 6-bit weight codes directly ("Qwen3.5 speed: prefill and decode
    parity with llama.cpp" #5305, child ticket #5221, against llama.cpp's
    quantised GEMV); the pages fix no rounding, so the oracle gives the exact
    value and the GPU's fp32 sums are compared within a tolerance."""
    return np.asarray(sa, np.float64)[:, None] * (qa.astype(np.float64) @ np.asarray(w, np.float64).T)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returned as float32."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = ((u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)) << np.uint64(16)
    return u.astype(np.uint32).view(np.float32)
