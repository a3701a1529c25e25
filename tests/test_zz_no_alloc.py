"""gdn_delta_rule_noalloc: the delta rule for callers that must not allocate
device memory (a plug-in whose host engine owns every device allocation, or a
loop that cannot afford cudaMalloc's implicit synchronisation).  Its scratch
is a static device array of the library, so the test checks it against the
allocating entry point, gdn_delta_rule, on two calls in a row: the second call
is shorter, so it runs over what the first one left in the shared array."""
import ctypes

import numpy as np
import pytest
import torch

from hybrid_gated_deltanet_q4k_gb300 import lib as gl
from hybrid_gated_deltanet_q4k_gb300 import synth
from oracle import layer as OL

from gpu_util import DEV, f16_dev, f32_dev, rel_l2, stream, sync

pytestmark = pytest.mark.gpu


def _inputs(spec, n, seed):
    rng = np.random.default_rng(seed)
    hk, hv, d = spec.n_qk_heads, spec.n_v_heads, spec.dk
    q = OL.l2norm_heads(rng.normal(size=(n, hk, d)), 1e-6) * d ** -0.5
    k = OL.l2norm_heads(rng.normal(size=(n, hk, d)), 1e-6)
    v = OL.silu(rng.normal(size=(n, hv, d)))
    qkv = np.concatenate([q.reshape(n, -1), k.reshape(n, -1), v.reshape(n, -1)], axis=1)
    la = rng.uniform(-0.5, 0, size=(n, hv)).astype(np.float32)
    b = (1 / (1 + np.exp(-rng.normal(size=(n, hv))))).astype(np.float32)
    s0 = rng.normal(0, 0.3, size=(hv, d, d)).astype(np.float32)
    return f16_dev(qkv), f32_dev(la), f32_dev(b), f32_dev(s0)


def _layer_struct(spec):
    dev = {k: f32_dev(np.zeros(64, np.float32)) for k in ("w_in", "w_out", "conv_w", "A_log", "dt_bias", "norm_w")}
    return gl.make_layer_struct(spec, dev), dev


@pytest.mark.parametrize("spec,lengths", [
    (synth.SPECS["h4096"], (700, 130)),
    (synth.LayerSpec("d4", 512, 2, 4, 128, 128, 0, "q4k", 6, ""), (1500, 65)),
])
def test_noalloc_matches_allocating_delta_rule(spec, lengths):
    L = gl.load(build=True)
    s, _keep = _layer_struct(spec)
    sp = ctypes.byref(s)
    for call, n in enumerate(lengths):
        qkv, la, b, s0 = _inputs(spec, n, seed=100 * call + n)
        o_ref = torch.empty(n, spec.c_v, dtype=torch.float16, device=DEV)
        st_ref = torch.empty_like(s0)
        nbytes = L.gdn_delta_rule_scratch_size(sp, n)
        assert nbytes <= gl.GDN_NOALLOC_SCRATCH_BYTES
        scratch = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
        L.gdn_delta_rule(sp, gl.ptr(qkv), gl.ptr(la), gl.ptr(b), n, gl.ptr(s0), gl.ptr(st_ref), gl.ptr(o_ref),
                         gl.ptr(scratch), nbytes, stream())
        o = torch.empty_like(o_ref)
        st = torch.empty_like(s0)
        L.gdn_delta_rule_noalloc(sp, gl.ptr(qkv), gl.ptr(la), gl.ptr(b), n, gl.ptr(s0), gl.ptr(st), gl.ptr(o), stream())
        sync(L)
        assert rel_l2(o.float().cpu().numpy(), o_ref.float().cpu().numpy()) <= 2e-3
        assert rel_l2(st.cpu().numpy(), st_ref.cpu().numpy()) <= 2e-3
        assert torch.equal(o, o_ref) and torch.equal(st, st_ref)   # same kernels, same order: same bits


def test_noalloc_rejects_more_tokens_than_its_scratch():
    L = gl.load(build=True)
    spec = synth.SPECS["h4096"]
    s, _keep = _layer_struct(spec)
    per_chunk = L.gdn_delta_rule_scratch_size(ctypes.byref(s), 64)
    fit = gl.GDN_NOALLOC_SCRATCH_BYTES // per_chunk * 64   # whole chunks of 64 tokens that fit the static array
    n = fit + 1
    assert L.gdn_delta_rule_scratch_size(ctypes.byref(s), fit) <= gl.GDN_NOALLOC_SCRATCH_BYTES
    assert L.gdn_delta_rule_scratch_size(ctypes.byref(s), n) > gl.GDN_NOALLOC_SCRATCH_BYTES
    buf = torch.zeros(16, dtype=torch.float32, device=DEV)
    r = L.gdn_delta_rule_noalloc(ctypes.byref(s), gl.ptr(buf), gl.ptr(buf), gl.ptr(buf), n, 0, gl.ptr(buf),
                                 gl.ptr(buf), stream(), check=False)
    assert r == gl.GDN_EINVAL
    assert f"at most {fit} tokens" in L.last_error()
