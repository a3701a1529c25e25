"""CPU checks of the C ABI: the library loads, exports every declared symbol,
its host-only encoder matches the oracle byte for byte, and argument checks
fail before touching a GPU."""
import ctypes

import numpy as np
import pytest

from hybrid_gated_deltanet_q4k_gb300 import lib as gl
from hybrid_gated_deltanet_q4k_gb300 import synth
from oracle import q4k


@pytest.fixture(scope="module")
def L():
    return gl.load(build=True)


def test_exports_every_declared_symbol(L):
    names = gl.header_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L.dll, n), n
    assert set(gl._SIGNATURES) == set(names)


def _pack(L, w):
    w = np.ascontiguousarray(w, np.float32)
    out = np.zeros((w.shape[0], w.shape[1] // 256 * 144), np.uint8)
    L.q4k_pack(gl.ptr(w), w.shape[0], w.shape[1], gl.ptr(out))
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_q4k_pack_matches_oracle_bytes(L, seed):
    rng = np.random.default_rng(seed)
    w = rng.normal(0, 0.02, size=(37, 1024)).astype(np.float32)
    w[3] = 0.0                      # zero row
    w[4] = -np.abs(w[4])            # all negative
    w[5] = np.abs(w[5])             # all positive
    w[6, :256] = 1e-6 * w[6, :256]  # tiny super-scales (fp16 subnormals)
    w[7, :32] = 7.5                 # constant sub-block
    assert np.array_equal(_pack(L, w), q4k.pack_q4k(w))


def test_q4k_pack_matches_oracle_on_layer_weights(L):
    spec = synth.SPECS["h1024"]
    layer = synth.make_layer(spec)
    w = layer["w_out"]
    assert np.array_equal(_pack(L, w), q4k.pack_q4k(w))


@pytest.mark.parametrize("seed", [0, 1])
def test_q6k_pack_matches_oracle_bytes(L, seed):
    from oracle import q6k
    rng = np.random.default_rng(seed + 100)
    w = rng.normal(0, 0.02, size=(21, 768)).astype(np.float32)
    w[2] = 0.0
    w[3] = -np.abs(w[3])
    w[4, :16] = 3.0                 # constant sub-block
    w[5, :256] = 1e-7 * w[5, :256]  # fp16 subnormal super-scale
    out = np.zeros((21, 3 * 210), np.uint8)
    L.q6k_pack(gl.ptr(w), 21, 768, gl.ptr(out))
    assert np.array_equal(out, q6k.pack_q6k(w))
    assert L.q6k_pack(gl.ptr(w), 21, 700, gl.ptr(out), check=False) == gl.GDN_EINVAL


def test_q4k_pack_rejects_bad_shapes(L):
    w = np.zeros((2, 300), np.float32)
    out = np.zeros(1000, np.uint8)
    assert L.q4k_pack(gl.ptr(w), 2, 300, gl.ptr(out), check=False) == gl.GDN_EINVAL
    assert L.q4k_pack(0, 2, 256, gl.ptr(out), check=False) == gl.GDN_EINVAL


def test_argument_checks_fail_without_gpu(L):
    spec = synth.SPECS["h2560"]
    s = gl.make_layer_struct(spec, {k: None for k in ("w_in", "w_out", "conv_w", "A_log", "dt_bias", "norm_w")})
    # null weights -> EINVAL, size query -> 0
    assert L.gdn_workspace_size(ctypes.byref(s), 512) == 0
    assert L.gdn_prefill(ctypes.byref(s), 0, 16, 0, 0, 0, 0, 0, 0, 0, check=False) == gl.GDN_EINVAL
    assert "NULL" in L.last_error()
    for name in ("w_in", "w_out", "conv_w", "A_log", "dt_bias", "norm_w"):
        setattr(s, name, 0x10000)   # fake, aligned addresses: never dereferenced by the checks below
    ws1 = L.gdn_workspace_size(ctypes.byref(s), 1)
    ws512 = L.gdn_workspace_size(ctypes.byref(s), 512)
    assert 0 < ws1 < ws512
    # the workspace grows linearly with the tokens per pass, in whole chunks of 64
    # (up to the 256-byte padding of each buffer)
    ws1024 = L.gdn_workspace_size(ctypes.byref(s), 1024)
    ws1536 = L.gdn_workspace_size(ctypes.byref(s), 1536)
    assert abs((ws1536 - ws1024) - (ws1024 - ws512)) <= 256 * 20
    # n_tokens <= 0, unsupported shapes, too small a workspace
    assert L.gdn_prefill(ctypes.byref(s), 0x10000, 0, 0, 0x10000, 0x10000, 0x10000, 0x10000, ws1, 0, check=False) == gl.GDN_EINVAL
    assert L.gdn_prefill(ctypes.byref(s), 0x10000, 8, 0, 0x10000, 0x10000, 0x10000, 0x10000, ws1 - 256, 0, check=False) == gl.GDN_ENOMEM
    s.conv_taps = 3
    assert L.gdn_workspace_size(ctypes.byref(s), 1) == 0
    s.conv_taps = 4
    s.n_v_heads = 24                 # not a multiple of 16 k heads
    assert L.gdn_prefill(ctypes.byref(s), 0x10000, 8, 0, 0x10000, 0x10000, 0x10000, 0x10000, ws512, 0, check=False) == gl.GDN_EINVAL
    s.n_v_heads = 32
    s.gate_log_a = 0x10000           # one gate pointer without the other
    assert L.gdn_workspace_size(ctypes.byref(s), 1) == 0
    s.gate_log_a = 0
    s.hidden = 2500                  # not a multiple of 256
    assert L.gdn_workspace_size(ctypes.byref(s), 1) == 0
    # stage entry points check their shapes before any launch
    assert L.q4k_deq_i8(0x10000, 4, 300, 0x10000, 0x10000, 0, check=False) == gl.GDN_EINVAL
    assert L.gdn_gemm_codes(0x10000, 0x10000, 0x10000, 0x10000, 128, 256, 100, 0x10000, 256, 256, 0, 0, 0, check=False) == gl.GDN_EINVAL
    assert L.gdn_quant_rows(0x10001, 4, 256, 0x10000, 0x10000, 0, check=False) == gl.GDN_EINVAL
