"""Seeded synthetic inputs for one Gated DeltaNet (GDN) prefill layer.

This module only draws random numbers: it holds none of the layer's own
arithmetic (no quantisation, no convolution, no recurrence).  Both the CUDA
library's tests and the CPU oracle take their inputs from here, so that the two
sides see the same bytes.

Workloads (sizes of Qwen3.5-family GDN layers; the pages measure on Qwen3.5
0.8B/4B/9B Q4_K_M GGUFs -- "CRUX parity spike: apr serve vs ollama on Qwen3.5",
part 2 tables -- whose trained weights are not used: every tensor below is
random, with the stated distribution):

* ``tiny_f32``  hidden 256, 2 q/k heads and 2 v heads of dim 64, N=64,
  fp32 weights (no quantisation), seed 0.
* ``h1024``     hidden 1024, 16 q/k heads x128, 16 v heads x128, N=512 (one
  ubatch of 512, the ubatch ollama uses), Q4_K weights, seed 1.
* ``h2560``     hidden 2560, 16 q/k heads x128, 32 v heads x128 (v heads share
  k heads 2:1), N=4096, Q4_K weights, seed 2.
* ``h4096``     hidden 4096, 16 q/k heads x128, 32 v heads x128, N=32768,
  Q4_K weights, log-decay ~ U(-0.5, 0), seed 3.
* ``extend``    the h2560 layer; 8 sequences with a 2048-token prefix and an
  extension of U[1, 4096] tokens each, seed 4.

Distributions: weight matrices and conv taps ~ N(0, 0.02); the gated-norm
weight ~ 1 + N(0, 0.02); A_log = dt_bias = 0; x ~ N(0, 1) (rounded to bf16 for
the Q4_K layers); gates drawn directly as a_t = exp(-softplus(u)), u ~ N(0, 1)
and b_t = sigmoid(N(0, 1)) (h4096: log a_t ~ U(-0.5, 0)).
"""
from __future__ import annotations

import dataclasses

import numpy as np

__all__ = ["LayerSpec", "SPECS", "make_layer", "make_tokens", "make_extend_case", "bf16_bits_to_f32"]


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    name: str
    hidden: int
    n_qk_heads: int
    n_v_heads: int
    dk: int
    dv: int
    n_tokens: int
    wtype: str  # "q4k" or "f32"
    seed: int
    gates: str  # "softplus_normal" or "uniform_logdecay"
    conv_taps: int = 4

    # Derived sizes (row counts of the fused input projection: q | k | v | z | beta | alpha).
    @property
    def c_qk(self) -> int:
        return self.n_qk_heads * self.dk

    @property
    def c_v(self) -> int:
        return self.n_v_heads * self.dv

    @property
    def c_conv(self) -> int:
        return 2 * self.c_qk + self.c_v

    @property
    def r_in(self) -> int:
        return 2 * self.c_qk + 2 * self.c_v + 2 * self.n_v_heads

    @property
    def workload(self) -> str:
        return (f"gdn_h{self.hidden}_qk{self.n_qk_heads}x{self.dk}_v{self.n_v_heads}x{self.dv}"
                f"_n{self.n_tokens}_{self.wtype}")


SPECS = {
    "tiny_f32": LayerSpec("tiny_f32", 256, 2, 2, 64, 64, 64, "f32", 0, "softplus_normal"),
    "h1024": LayerSpec("h1024", 1024, 16, 16, 128, 128, 512, "q4k", 1, "softplus_normal"),
    "h2560": LayerSpec("h2560", 2560, 16, 32, 128, 128, 4096, "q4k", 2, "softplus_normal"),
    "h4096": LayerSpec("h4096", 4096, 16, 32, 128, 128, 32768, "q4k", 3, "uniform_logdecay"),
    "extend": LayerSpec("extend", 2560, 16, 32, 128, 128, 2048, "q4k", 4, "softplus_normal"),
}


def _round_bf16_inplace(x32: np.ndarray) -> np.ndarray:
    """Round finite float32 values to the nearest-even bf16, in place, in row
    blocks (input recipe only); returns the bf16 bit patterns."""
    u = x32.reshape(-1).view(np.uint32)
    bits = np.empty(u.shape, np.uint16)
    step = 1 << 22
    tmp = np.empty(min(step, u.size), np.uint32)
    for i in range(0, u.size, step):
        seg = u[i:i + step]
        t = tmp[:seg.size]
        np.right_shift(seg, 16, out=t)
        t &= 1
        t += 0x7FFF
        seg += t
        seg &= 0xFFFF0000
        np.right_shift(seg, 16, out=t)
        bits[i:i + step] = t
    return bits.reshape(x32.shape)


def _to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Nearest-even bf16 bit pattern of finite float32 input values (input recipe only)."""
    return _round_bf16_inplace(np.array(x32, dtype=np.float32, copy=True))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact float32 value of bf16 bit patterns."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def make_layer(spec: LayerSpec, seed: int | None = None) -> dict:
    """Random layer parameters in float32 (weights are quantised later, by each side)."""
    rng = np.random.default_rng(spec.seed if seed is None else seed)
    f32 = np.float32
    w_in = rng.standard_normal((spec.r_in, spec.hidden), dtype=f32) * f32(0.02)
    w_out = rng.standard_normal((spec.hidden, spec.c_v), dtype=f32) * f32(0.02)
    conv_w = rng.standard_normal((spec.c_conv, spec.conv_taps), dtype=f32) * f32(0.02)
    norm_w = f32(1.0) + rng.standard_normal(spec.dv, dtype=f32) * f32(0.02)
    return {
        "w_in": w_in,
        "w_out": w_out,
        "conv_w": conv_w,
        "A_log": np.zeros(spec.n_v_heads, np.float32),
        "dt_bias": np.zeros(spec.n_v_heads, np.float32),
        "norm_w": norm_w,
    }


def make_tokens(spec: LayerSpec, n_tokens: int, seed: int) -> dict:
    """x [N, hidden] and directly drawn gates log_a, b [N, Hv].

    For Q4_K layers x is returned both as bf16 bit patterns (``x_bits``) and as
    the exact float32 value of those patterns (``x``)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n_tokens, spec.hidden), dtype=np.float32)
    hv = spec.n_v_heads
    if spec.gates == "uniform_logdecay":
        log_a = rng.uniform(-0.5, 0.0, size=(n_tokens, hv))
    else:
        u = rng.normal(0.0, 1.0, size=(n_tokens, hv))
        log_a = -np.logaddexp(0.0, u)  # a = exp(-softplus(u))
    b = 1.0 / (1.0 + np.exp(-rng.normal(0.0, 1.0, size=(n_tokens, hv))))
    out = {"log_a": log_a.astype(np.float32), "b": b.astype(np.float32)}
    if spec.wtype == "q4k":
        out["x_bits"] = _round_bf16_inplace(x)   # x now holds the bf16 values
        out["x"] = x
    else:
        out["x"] = x
    return out


def make_extend_case(spec: LayerSpec, n_seqs: int = 8, prefix: int = 2048, max_ext: int = 4096) -> list:
    """Session-extend workload: per sequence a prefix and an extension length.

    Returns a list of dicts with the prompt tokens of the full concatenation
    (prefix + extension) and the split point."""
    rng = np.random.default_rng(spec.seed)
    ext = rng.integers(1, max_ext + 1, size=n_seqs)
    cases = []
    for i in range(n_seqs):
        toks = make_tokens(spec, prefix + int(ext[i]), seed=spec.seed * 1000 + i)
        toks["prefix"] = prefix
        toks["extension"] = int(ext[i])
        cases.append(toks)
    return cases


def make_attention(nq: int, nk: int, hq: int, hkv: int, d: int, seed: int, q_gain: float = 1.0) -> dict:
    """Inputs of the full-attention prefill: q [nq, hq, d], k and v [nk, hkv, d]
    ~ N(0, 1) (q times q_gain: a larger gain makes the softmax peakier), rounded
    to bf16; returned as bit patterns (``*_bits``) and their exact float32
    values."""
    rng = np.random.default_rng(seed)
    out = {}
    for name, shape, gain in (("q", (nq, hq, d), q_gain), ("k", (nk, hkv, d), 1.0), ("v", (nk, hkv, d), 1.0)):
        x = rng.standard_normal(shape, dtype=np.float32)
        if gain != 1.0:
            x *= np.float32(gain)
        out[name + "_bits"] = _round_bf16_inplace(x)
        out[name] = x
    return out
