"""Causal grouped-query attention prefill (gdn_attn_prefill) against the oracle.

Tolerance, from the arithmetic: the inputs are the same bf16 values on both
sides; the GPU's scores and sums are fp32, its probabilities enter the second
product rounded to bf16 (2^-9 relative each, independent) and the output is
rounded to bf16 (2^-9 relative); relative L2 <= 4e-3 over the output, every
element within 2^-6 of its row's largest magnitude.  Full size (32768 tokens,
16 query heads over 4 key/value heads of 256) is checked on sampled rows the
oracle computes one by one.
"""
import numpy as np
import pytest
import torch

from hybrid_gated_deltanet_q4k_gb300 import lib as gl
from hybrid_gated_deltanet_q4k_gb300 import synth
from oracle import attention as OA

from gpu_util import DEV, rel_l2, stream, sync

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    return gl.load(build=True)


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def _run(L, inp, nq, nk, hq, hkv, d, scale=0.0):
    q, k, v = _dev(inp["q_bits"]), _dev(inp["k_bits"]), _dev(inp["v_bits"])
    o = torch.empty(nq, hq, d, dtype=torch.bfloat16, device=DEV)
    nbytes = L.gdn_attn_workspace_size(nk, hkv, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    L.gdn_attn_prefill(gl.ptr(q), gl.ptr(k), gl.ptr(v), nq, nk, hq, hkv, d, scale, gl.ptr(o), gl.ptr(ws), nbytes, stream())
    sync(L)
    return o.float().cpu().numpy()


def _check(got, ref):
    assert rel_l2(got, ref) <= 4e-3
    rowmax = np.abs(ref).max(axis=-1, keepdims=True)
    assert np.all(np.abs(got - ref) <= 2.0 ** -6 * rowmax + 1e-6)


@pytest.mark.parametrize("nq,nk,hq,hkv,d,gain", [
    (200, 200, 4, 2, 64, 1.0), (300, 300, 2, 1, 128, 1.0), (130, 130, 2, 2, 256, 1.0),
    (70, 333, 4, 1, 128, 1.0),        # queries extending 263 held keys
    (1, 100, 2, 2, 128, 1.0), (1, 1, 2, 1, 64, 1.0),
    (257, 257, 2, 1, 128, 6.0),       # peaked softmax: the running maximum is raised often
    (513, 700, 8, 2, 256, 3.0),
])
def test_attention_matches_oracle(L, nq, nk, hq, hkv, d, gain):
    inp = synth.make_attention(nq, nk, hq, hkv, d, seed=nq + nk + d, q_gain=gain)
    got = _run(L, inp, nq, nk, hq, hkv, d)
    _check(got, OA.attention(inp["q"], inp["k"], inp["v"]))


def test_attention_explicit_scale_and_extend(L):
    """An explicit scale, and queries extending held keys equal the last rows of
    the full prefill (the same computation per row)."""
    nk, hq, hkv, d = 400, 4, 2, 128
    inp = synth.make_attention(nk, nk, hq, hkv, d, seed=9)
    full = _run(L, inp, nk, nk, hq, hkv, d, scale=0.05)
    tail_inp = dict(inp, q_bits=inp["q_bits"][300:], q=inp["q"][300:])
    tail = _run(L, tail_inp, 100, nk, hq, hkv, d, scale=0.05)
    assert np.array_equal(tail, full[300:])
    _check(full, OA.attention(inp["q"], inp["k"], inp["v"], scale=0.05))


def test_attention_full_size_sampled_rows(L):
    nq = nk = 32768
    hq, hkv, d = 16, 4, 256
    inp = synth.make_attention(nq, nk, hq, hkv, d, seed=3)
    got = _run(L, inp, nq, nk, hq, hkv, d)
    rng = np.random.default_rng(0)
    rows = sorted(set([0, 1, 127, 128, 4095, 32767] + list(rng.integers(0, nq, size=10))))
    for i in rows:
        for h in (0, 5, 15):
            g = h // (hq // hkv)
            ref = OA.attention(inp["q"][i:i + 1, h:h + 1], inp["k"][: i + 1, g:g + 1], inp["v"][: i + 1, g:g + 1])
            _check(got[i:i + 1, h:h + 1], ref)


def test_attention_argument_checks(L):
    z = torch.zeros(64, 2, 64, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    bad = [(64, 64, 2, 1, 96), (64, 32, 2, 2, 64), (64, 64, 3, 2, 64), (0, 64, 2, 2, 64)]
    for nq, nk, hq, hkv, d in bad:
        r = L.gdn_attn_prefill(gl.ptr(z), gl.ptr(z), gl.ptr(z), nq, nk, hq, hkv, d, 0.0, gl.ptr(z), gl.ptr(ws),
                               ws.numel(), stream(), check=False)
        assert r == gl.GDN_EINVAL, (nq, nk, hq, hkv, d)
    r = L.gdn_attn_prefill(gl.ptr(z), gl.ptr(z), gl.ptr(z), 64, 64, 2, 2, 64, 0.0, gl.ptr(z), gl.ptr(ws), 16, stream(),
                           check=False)
    assert r == gl.GDN_ENOMEM
