"""Stage-by-stage parity of the CUDA kernels with the oracle, through the C ABI.

Integer and byte work (Q4_K decode to int8 rows, activation quantisation, the
integer product and its fp32 rescale) must be bit-exact.  Floating-point
stages are fed the same inputs as the oracle and compared within tolerances
derived from their arithmetic:
  * conv + SiLU + L2 norm (fp16 out, the recurrence's tensor-core operand
    type): each element within 2^-11 + 3e-5 relative of the fp64 value (the
    fp16 rounding, plus a few fp32 roundings in the 4-tap sum, the
    exponential, the 128-term norm and the reciprocal square root) plus 1e-6
    of the tensor's largest magnitude (cancellation in the tap sum);
  * gated delta rule (fp32 state, chunked): relative L2 <= 2e-3 for o and the
    final state;
  * gated RMSNorm: fp32 output within relative L2 1e-5; int8 codes within
    one step of the oracle's, the scale within 1e-5.
"""
import ctypes

import numpy as np
import pytest
import torch

from hybrid_gated_deltanet_q4k_gb300 import lib as gl
from hybrid_gated_deltanet_q4k_gb300 import synth
from oracle import layer as OL
from oracle import q4k, q6k, quant

from gpu_util import DEV, bf16_dev, bf16_host_f32, f16_codes, f16_dev, f16_round, f32_dev, rel_l2, stream, sync

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return gl.load(build=True)


# ------------------------------------------------------------------ step 1a

@pytest.mark.parametrize("rows,cols", [(1, 256), (516, 256), (1024, 2048), (8224, 1024), (4096, 4096),
                                       (12352, 2560), (5, 16384)])
def test_q4k_deq_bit_exact(L, rows, cols):
    rng = np.random.default_rng(rows * 7 + cols)
    w = rng.normal(0, 0.02, size=(rows, cols)).astype(np.float32)
    if rows > 4:
        w[1] = 0.0
        w[2] = 0.37
        w[3, ::3] *= 40.0
    blocks = q4k.pack_q4k(w)
    ref_q, ref_s = quant.quant_rows_i8(q4k.unpack_q4k(blocks, rows, cols))
    b = torch.from_numpy(blocks).to(DEV)
    q = torch.empty(rows, cols, dtype=torch.int8, device=DEV)
    s = torch.empty(rows, dtype=torch.float32, device=DEV)
    L.q4k_deq_i8(gl.ptr(b), rows, cols, gl.ptr(q), gl.ptr(s), stream())
    codes = torch.empty(rows, cols, dtype=torch.float16, device=DEV)
    s2 = torch.empty(rows, dtype=torch.float32, device=DEV)
    L.gdn_q4k_deq_codes(gl.ptr(b), rows, cols, gl.ptr(codes), gl.ptr(s2), stream())
    sync(L)
    assert np.array_equal(q.cpu().numpy(), ref_q)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(f16_codes(codes), ref_q.astype(np.int64))
    assert np.array_equal(s2.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))


@pytest.mark.parametrize("rows,cols", [(1, 256), (7, 512), (1024, 2048), (4096, 4096), (3, 16384), (12352, 256)])
def test_q6k_deq_bit_exact(L, rows, cols):
    """Q6_K rows (the fused dequant's second format) decode and quantise to
    the oracle's int8 codes and row scales byte for byte."""
    rng = np.random.default_rng(rows * 5 + cols)
    w = rng.normal(0, 0.02, size=(rows, cols)).astype(np.float32)
    if rows > 4:
        w[1] = 0.0
        w[2] = -0.37
        w[3, ::5] *= 60.0
    blocks = q6k.pack_q6k(w)
    ref_q, ref_s = quant.quant_rows_i8(q6k.unpack_q6k(blocks, rows, cols))
    b = torch.from_numpy(blocks).to(DEV)
    q = torch.empty(rows, cols, dtype=torch.int8, device=DEV)
    s = torch.empty(rows, dtype=torch.float32, device=DEV)
    L.q6k_deq_i8(gl.ptr(b), rows, cols, gl.ptr(q), gl.ptr(s), stream())
    codes = torch.empty(rows, cols, dtype=torch.float16, device=DEV)
    s2 = torch.empty(rows, dtype=torch.float32, device=DEV)
    L.gdn_q6k_deq_codes(gl.ptr(b), rows, cols, gl.ptr(codes), gl.ptr(s2), stream())
    sync(L)
    assert np.array_equal(q.cpu().numpy(), ref_q)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(f16_codes(codes), ref_q.astype(np.int64))
    assert np.array_equal(s2.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))


def test_q6k_deq_extreme_codes(L):
    """Blocks with every code at -32 or 31 and scales at -128 / 127 (the ends
    of both fields) and a row holding one nonzero weight."""
    rng = np.random.default_rng(2)
    rows, cols = 6, 1024
    raw = rng.integers(0, 256, size=(rows, cols // 256, 210), dtype=np.uint8)
    raw[:, :, 208:210] = np.array([2.0 ** -9], np.float16).view(np.uint8)   # finite d everywhere
    raw[0, :, :192] = 0                                                     # codes 0: q = -32
    raw[0, :, 192:208] = np.uint8(0x80)                                     # scales -128
    raw[1, :, :192] = 0xFF                                                  # codes 63: q = 31
    raw[1, :, 192:208] = 127
    raw[2, :, 128:192] = 0xAA                                               # q = 0 except one weight
    raw[2, :, :128] = 0
    raw[2, 1, 5] = 3                                                        # weight 5 of superblock 1: q = 3
    raw[2, 1, 192] = 5                                                      # its scale
    blocks = raw.reshape(rows, -1)
    ref_q, ref_s = quant.quant_rows_i8(q6k.unpack_q6k(blocks, rows, cols))
    b = torch.from_numpy(blocks.copy()).to(DEV)
    q = torch.empty(rows, cols, dtype=torch.int8, device=DEV)
    s = torch.empty(rows, dtype=torch.float32, device=DEV)
    L.q6k_deq_i8(gl.ptr(b), rows, cols, gl.ptr(q), gl.ptr(s), stream())
    sync(L)
    assert np.array_equal(q.cpu().numpy(), ref_q)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert np.count_nonzero(ref_q[2]) == 1


# ------------------------------------------------------------------ step 1b

@pytest.mark.parametrize("rows,cols", [(1, 8), (300, 1024), (77, 2560), (33, 4096), (3, 16384), (4096, 4096)])
def test_quant_rows_bit_exact(L, rows, cols):
    rng = np.random.default_rng(cols)
    # per-row magnitudes over six decades: many rows, so the codes that fall near a
    # rounding tie of x / scale (the fast quantiser's exact fallback) are covered
    x = (rng.normal(0, 1, size=(rows, cols)) * 10.0 ** rng.uniform(-3, 3, size=(rows, 1))).astype(np.float32)
    if rows >= 3:
        x[0] = 0.0
        x[1, :] = 0.0
        x[1, 0] = 127.0
        x[1, 1:9] = [2.5, 3.5, -2.5, 0.5, -0.5, 1.5, 126.5, -126.5]   # ties at scale 1: nearest even
    bits = synth._to_bf16_bits(x)
    x32 = synth.bf16_bits_to_f32(bits)
    ref_q, ref_s = quant.quant_rows_i8(x32)
    xd = bf16_dev(bits)
    codes = torch.empty(rows, cols, dtype=torch.float16, device=DEV)
    s = torch.empty(rows, dtype=torch.float32, device=DEV)
    L.gdn_quant_rows(gl.ptr(xd), rows, cols, gl.ptr(codes), gl.ptr(s), stream())
    sync(L)
    assert np.array_equal(f16_codes(codes), ref_q.astype(np.int64))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))


# ------------------------------------------------------------------ steps 1c, 5

def _run_gemm(L, qa, sa, qb, sb, n_bf16):
    M, K = qa.shape
    N = qb.shape[0]
    a = torch.from_numpy(qa.astype(np.float16)).to(DEV)
    b = torch.from_numpy(qb.astype(np.float16)).to(DEV)
    sad, sbd = f32_dev(sa), f32_dev(sb)
    ob = torch.zeros(M, max(n_bf16, 1), dtype=torch.bfloat16, device=DEV)
    of = torch.zeros(M, max(N - n_bf16, 1), dtype=torch.float32, device=DEV)
    L.gdn_gemm_codes(gl.ptr(a), gl.ptr(sad), gl.ptr(b), gl.ptr(sbd), M, N, K, gl.ptr(ob), max(n_bf16, 1), n_bf16,
                     gl.ptr(of), max(N - n_bf16, 1), stream())
    sync(L)
    return bf16_host_f32(ob)[:, :n_bf16], of.cpu().numpy()[:, :N - n_bf16]


@pytest.mark.parametrize("M,N,K", [(1, 256, 256), (127, 300, 1024), (200, 8224, 1024), (513, 12352, 2560),
                                   (129, 2560, 4096), (64, 4096, 4096), (300, 130, 64), (256, 512, 2048)])
def test_gemm_codes_bit_exact(L, M, N, K):
    rng = np.random.default_rng(M + N + K)
    qa = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    qb = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
    sa = rng.uniform(1e-3, 1e-1, size=M).astype(np.float32)
    sb = rng.uniform(1e-4, 1e-2, size=N).astype(np.float32)
    n_bf16 = N - 64 if N > 256 else N
    yb, yf = _run_gemm(L, qa, sa, qb, sb, n_bf16)
    ref = quant.gemm_q8(qa, sa, qb, sb)
    assert np.array_equal(yb.view(np.uint32), quant.bf16_round(ref[:, :n_bf16]).view(np.uint32))
    assert np.array_equal(yf.view(np.uint32), ref[:, n_bf16:].view(np.uint32))


def test_gemm_exact_beyond_fp32_integer_range(L):
    """Sums up to 4096 * 127^2 > 2^24: exact only because each 1024-term segment is."""
    M, N, K = 130, 260, 4096
    qa = np.full((M, K), 127, np.int8)
    qa[1::2] = -127
    qb = np.full((N, K), 127, np.int8)
    qb[:, 1::7] = -127
    qb[5, :] = 1
    sa = np.ones(M, np.float32)
    sb = np.ones(N, np.float32)
    _, yf = _run_gemm(L, qa, sa, qb, sb, 0)
    acc = quant.int_matmul_exact(qa, qb)
    assert np.abs(acc).max() > 2 ** 24
    assert np.array_equal(yf, acc.astype(np.float32))


def test_gemm_f32(L):
    rng = np.random.default_rng(9)
    M, N, K = 70, 516, 256
    a = rng.normal(size=(M, K)).astype(np.float32)
    b = rng.normal(0, 0.02, size=(N, K)).astype(np.float32)
    ad, bd = f32_dev(a), f32_dev(b)
    ob = torch.zeros(M, 512, dtype=torch.bfloat16, device=DEV)
    of = torch.zeros(M, 4, dtype=torch.float32, device=DEV)
    L.gdn_gemm_f32(gl.ptr(ad), gl.ptr(bd), M, N, K, gl.ptr(ob), 512, 512, gl.ptr(of), 4, stream())
    sync(L)
    ref = a.astype(np.float64) @ b.astype(np.float64).T
    assert rel_l2(of.cpu().numpy(), ref[:, 512:]) < 1e-6
    got = bf16_host_f32(ob)
    assert np.all(np.abs(got - ref[:, :512]) <= 2 ** -8 * np.abs(ref[:, :512]) + 1e-6)


# ------------------------------------------------------------------ step 2

def _layer(spec, L_, gates=False):
    layer = synth.make_layer(spec, seed=spec.seed + 100)
    dev = {k: f32_dev(layer[k]) for k in ("conv_w", "A_log", "dt_bias", "norm_w")}
    dev["w_in"] = dev["w_out"] = f32_dev(np.zeros(16, np.float32))   # unused by the stage calls
    layer["A_log"] = np.random.default_rng(1).normal(0, 0.5, spec.n_v_heads).astype(np.float32)
    layer["dt_bias"] = np.random.default_rng(2).normal(0, 0.5, spec.n_v_heads).astype(np.float32)
    dev["A_log"], dev["dt_bias"] = f32_dev(layer["A_log"]), f32_dev(layer["dt_bias"])
    s = gl.make_layer_struct(spec, dev)
    return layer, dev, s


CONV_SPECS = [synth.SPECS["tiny_f32"], synth.SPECS["h2560"], synth.LayerSpec("s", 512, 2, 4, 128, 128, 0, "q4k", 5, "")]


@pytest.mark.parametrize("spec", CONV_SPECS, ids=lambda s: s.name)
@pytest.mark.parametrize("n", [1, 2, 3, 5, 64, 65, 130])
def test_conv_stage(L, spec, n):
    layer, dev, s = _layer(spec, L)
    rng = np.random.default_rng(n)
    nb = 2 * spec.c_qk + 2 * spec.c_v
    bits = synth._to_bf16_bits(rng.normal(0, 1.3, size=(n, nb)).astype(np.float32))
    raw = synth.bf16_bits_to_f32(bits)
    tail = synth.bf16_bits_to_f32(synth._to_bf16_bits(rng.normal(0, 1.3, size=(spec.c_conv, 3)).astype(np.float32)))
    ba = rng.normal(0, 1, size=(n, 2 * spec.n_v_heads)).astype(np.float32)
    qkvz, taild, bad = bf16_dev(bits), f32_dev(tail), f32_dev(ba)
    qkv = torch.empty(n, spec.c_conv, dtype=torch.float16, device=DEV)
    la = torch.empty(n, spec.n_v_heads, dtype=torch.float32, device=DEV)
    bb = torch.empty_like(la)
    L.gdn_conv(ctypes.byref(s), gl.ptr(qkvz), nb, n, gl.ptr(taild), gl.ptr(bad), 2 * spec.n_v_heads, gl.ptr(qkv),
               gl.ptr(la), gl.ptr(bb), stream())
    L.gdn_conv_state_update(ctypes.byref(s), gl.ptr(qkvz), nb, n, gl.ptr(taild), stream())
    sync(L)
    p = dict(n_qk_heads=spec.n_qk_heads, n_v_heads=spec.n_v_heads, dk=spec.dk, dv=spec.dv, conv_w=layer["conv_w"],
             eps_l2=1e-6, q_scale=spec.dk ** -0.5, wtype=spec.wtype, hidden=spec.hidden)
    q, k, v, new_tail = OL.conv_stage(p, raw[:, :spec.c_conv], tail)
    ref = np.concatenate([q.reshape(n, -1), k.reshape(n, -1), v.reshape(n, -1)], axis=1)
    got = qkv.float().cpu().numpy()
    # fp16 rounding (half an ulp: 2^-11 relative, 2^-25 absolute below the normal
    # range) on top of the fp32 arithmetic
    bound = (2 ** -11 + 3e-5) * np.abs(ref) + 1e-6 * np.abs(ref).max()
    assert np.all(np.abs(got - ref) <= bound)
    assert np.array_equal(taild.cpu().numpy(), new_tail.astype(np.float32))
    rla, rb = OL.gates(ba[:, spec.n_v_heads:], ba[:, :spec.n_v_heads], layer["A_log"], layer["dt_bias"])
    assert rel_l2(la.cpu().numpy(), rla) < 1e-5
    assert rel_l2(bb.cpu().numpy(), rb) < 1e-6


def test_conv_reports_fp16_overflow(L):
    """A conv output beyond the fp16 range (|y| > 65504) is reported once as
    GDN_ERANGE by the next status read, which also clears it."""
    spec = CONV_SPECS[2]
    layer, dev, s = _layer(spec, L)
    n = 70
    rng = np.random.default_rng(5)
    nb = 2 * spec.c_qk + 2 * spec.c_v
    x = rng.normal(0, 1.0, size=(n, nb)).astype(np.float32)
    # the v channel whose filter taps sum furthest from zero, driven with a constant
    # of that sum's sign: SiLU(conv) = 3e6 |sum| once all taps see it, far above 65504
    vch = 2 * spec.c_qk + np.arange(spec.c_v)
    wsum = np.asarray(layer["conv_w"], np.float64).reshape(spec.c_conv, -1)[vch].sum(axis=1)
    c = int(np.argmax(np.abs(wsum)))
    assert abs(wsum[c]) > 0.05
    x[:, vch[c]] = 3.0e6 * np.sign(wsum[c])
    qkvz, taild = bf16_dev(synth._to_bf16_bits(x)), f32_dev(np.zeros((spec.c_conv, 3), np.float32))
    bad = f32_dev(np.zeros((n, 2 * spec.n_v_heads), np.float32))
    qkv = torch.empty(n, spec.c_conv, dtype=torch.float16, device=DEV)
    la = torch.empty(n, spec.n_v_heads, dtype=torch.float32, device=DEV)
    bb = torch.empty_like(la)
    L.gdn_conv(ctypes.byref(s), gl.ptr(qkvz), nb, n, gl.ptr(taild), gl.ptr(bad), 2 * spec.n_v_heads, gl.ptr(qkv),
               gl.ptr(la), gl.ptr(bb), stream())
    assert L.gdn_sync_status(stream(), check=False) == gl.GDN_ERANGE
    assert "fp16" in L.last_error() or "range" in L.last_error()
    assert L.gdn_sync_status(stream(), check=False) == gl.GDN_OK


# ------------------------------------------------------------------ step 3

def _delta_inputs(spec, n, rng):
    hk, hv, d = spec.n_qk_heads, spec.n_v_heads, spec.dk
    q = OL.l2norm_heads(rng.normal(size=(n, hk, d)), 1e-6) * d ** -0.5
    k = OL.l2norm_heads(rng.normal(size=(n, hk, d)), 1e-6)
    v = OL.silu(rng.normal(0, 1, size=(n, hv, d)))
    # the recurrence consumes q, k, v in fp16, as gdn_conv writes them
    qkv = f16_round(np.concatenate([q.reshape(n, -1), k.reshape(n, -1), v.reshape(n, -1)], axis=1))
    vals = qkv.astype(np.float64)
    c = spec.c_qk
    qe = OL.expand_kv_heads(vals[:, :c].reshape(n, hk, d), hv)
    ke = OL.expand_kv_heads(vals[:, c:2 * c].reshape(n, hk, d), hv)
    ve = vals[:, 2 * c:].reshape(n, hv, d)
    if spec.gates == "uniform_logdecay":
        la = rng.uniform(-0.5, 0, size=(n, hv))
    else:
        la = -np.logaddexp(0, rng.normal(size=(n, hv)))
    b = 1 / (1 + np.exp(-rng.normal(size=(n, hv))))
    return qkv, qe, ke, ve, la.astype(np.float32), b.astype(np.float32)


DELTA_SPECS = [synth.SPECS["tiny_f32"], synth.LayerSpec("d4", 512, 2, 4, 128, 128, 0, "q4k", 6, "softplus_normal"),
               synth.LayerSpec("d4u", 512, 2, 4, 128, 128, 0, "q4k", 7, "uniform_logdecay")]


@pytest.mark.parametrize("spec", DELTA_SPECS, ids=lambda s: s.name)
@pytest.mark.parametrize("n,with_state", [(1, True), (63, False), (64, True), (65, True), (200, False),
                                          (513, True), (2000, True), (8300, True)])
def test_delta_rule_stage(L, spec, n, with_state):
    _, dev, s = _layer(spec, L)
    rng = np.random.default_rng(1000 + n)
    qkv_h, qe, ke, ve, la, b = _delta_inputs(spec, n, rng)
    S0 = rng.normal(0, 0.3, size=(spec.n_v_heads, spec.dv, spec.dk)).astype(np.float32) if with_state else None
    qkv, lad, bd = f16_dev(qkv_h), f32_dev(la), f32_dev(b)
    sin = f32_dev(S0) if with_state else None
    sout = torch.empty(spec.n_v_heads, spec.dv, spec.dk, dtype=torch.float32, device=DEV)
    o = torch.empty(n, spec.c_v, dtype=torch.float16, device=DEV)
    nbytes = L.gdn_delta_rule_scratch_size(ctypes.byref(s), n)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    L.gdn_delta_rule(ctypes.byref(s), gl.ptr(qkv), gl.ptr(lad), gl.ptr(bd), n, gl.ptr(sin), gl.ptr(sout), gl.ptr(o),
                     gl.ptr(scratch), nbytes, stream())
    sync(L)
    S0r = S0 if with_state else np.zeros((spec.n_v_heads, spec.dv, spec.dk))
    ro, rS = OL.gated_delta_rule(qe, ke, ve, la, b, S0r)
    assert rel_l2(o.float().cpu().numpy(), ro.reshape(n, -1)) <= 2e-3
    assert rel_l2(sout.cpu().numpy(), rS) <= 2e-3


def test_delta_rule_decay_paths(L):
    """The prep evaluates a chunk's decays e^{gamma_i - gamma_j} as e^{gamma_i}
    e^{-gamma_j} when the chunk's whole decay gamma_C is at least -64 and by
    their own exponentials below that.  Value heads here decay by 0.1 to 2 per
    token (gamma_C from -6 to -128 over a chunk), so both ways are taken, also
    by the two value heads of one key head within a CTA; o and the state match
    the fp64 recurrence either way."""
    spec = DELTA_SPECS[1]
    _, dev, s = _layer(spec, L)
    rng = np.random.default_rng(4242)
    n = 1000
    qkv_h, qe, ke, ve, _, b = _delta_inputs(spec, n, rng)
    rate = np.array([0.1, 2.0, 0.9, 1.1])[: spec.n_v_heads]          # per value head: gamma_C ~ -64 * rate
    la = (-rate[None, :] * rng.uniform(0.8, 1.2, size=(n, spec.n_v_heads))).astype(np.float32)
    S0 = rng.normal(0, 0.3, size=(spec.n_v_heads, spec.dv, spec.dk)).astype(np.float32)
    qkv, lad, bd = f16_dev(qkv_h), f32_dev(la), f32_dev(b)
    sout = torch.empty(spec.n_v_heads, spec.dv, spec.dk, dtype=torch.float32, device=DEV)
    o = torch.empty(n, spec.c_v, dtype=torch.float16, device=DEV)
    nbytes = L.gdn_delta_rule_scratch_size(ctypes.byref(s), n)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    L.gdn_delta_rule(ctypes.byref(s), gl.ptr(qkv), gl.ptr(lad), gl.ptr(bd), n, gl.ptr(f32_dev(S0)), gl.ptr(sout),
                     gl.ptr(o), gl.ptr(scratch), nbytes, stream())
    sync(L)
    whole = n - n % 64
    gamma_c = la[:whole].astype(np.float64).reshape(whole // 64, 64, spec.n_v_heads).sum(axis=1)
    assert (gamma_c >= -64).any() and (gamma_c < -64).any()
    ro, rS = OL.gated_delta_rule(qe, ke, ve, la, b, S0)
    assert rel_l2(o.float().cpu().numpy(), ro.reshape(n, -1)) <= 2e-3
    assert rel_l2(sout.cpu().numpy(), rS) <= 2e-3


def test_delta_rule_segments_bitwise(L):
    """Inputs longer than 64 chunks run as token segments (the prep of the next
    segment beside the state pass of the current one) with the fp32 state
    carried between them: one call over 8300 tokens (three segments) gives the
    same bits as a call over the first 4096 tokens (one segment) followed by
    one over the rest (two segments)."""
    spec = DELTA_SPECS[1]
    _, dev, s = _layer(spec, L)
    rng = np.random.default_rng(79)
    n, n1 = 8300, 4096
    qkv_h, qe, ke, ve, la, b = _delta_inputs(spec, n, rng)
    S0 = rng.normal(0, 0.3, size=(spec.n_v_heads, spec.dv, spec.dk)).astype(np.float32)
    qkv, lad, bd = f16_dev(qkv_h), f32_dev(la), f32_dev(b)

    def run(lo, hi, sin, sout, o):
        m = hi - lo
        nbytes = L.gdn_delta_rule_scratch_size(ctypes.byref(s), m)
        scratch = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
        L.gdn_delta_rule(ctypes.byref(s), gl.ptr(qkv[lo:hi]), gl.ptr(lad[lo:hi]), gl.ptr(bd[lo:hi]), m, gl.ptr(sin),
                         gl.ptr(sout), gl.ptr(o[lo:hi]), gl.ptr(scratch), nbytes, stream())
        sync(L)

    o_one = torch.empty(n, spec.c_v, dtype=torch.float16, device=DEV)
    st_one = torch.empty(spec.n_v_heads, spec.dv, spec.dk, dtype=torch.float32, device=DEV)
    run(0, n, f32_dev(S0), st_one, o_one)
    o_two = torch.empty_like(o_one)
    st_two = f32_dev(S0)
    run(0, n1, st_two, st_two, o_two)
    run(n1, n, st_two, st_two, o_two)
    assert torch.equal(o_one, o_two) and torch.equal(st_one, st_two)
    ro, rS = OL.gated_delta_rule(qe, ke, ve, la, b, S0)
    assert rel_l2(o_one.float().cpu().numpy(), ro.reshape(n, -1)) <= 2e-3
    assert rel_l2(st_one.cpu().numpy(), rS) <= 2e-3


@pytest.mark.parametrize("spec", DELTA_SPECS[:2], ids=lambda s: s.name)
def test_delta_rule_wait_runs_out_then_recovers(L, spec):
    """Fail closed on a bounded device wait (sparkinfer PR #464, eval-bot
    thread: an infrastructure failure must surface as a failure, not as a
    result).  gdn_test_delta_wait_timeout runs the delta rule's prep with its
    [Q; K] copy never issued and a 1 ms limit on the wait for it: the kernel
    records the timeout, frees its tensor memory and returns, nothing faults,
    gdn_sync_status reports GDN_ETIMEOUT once, and the next gdn_delta_rule
    call runs normally and matches the oracle."""
    _, dev, s = _layer(spec, L)
    rng = np.random.default_rng(91)
    n = 200
    qkv_h, qe, ke, ve, la, b = _delta_inputs(spec, n, rng)
    qkv, lad, bd = f16_dev(qkv_h), f32_dev(la), f32_dev(b)
    nbytes = L.gdn_delta_rule_scratch_size(ctypes.byref(s), n)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    args = (ctypes.byref(s), gl.ptr(qkv), gl.ptr(lad), gl.ptr(bd), n, gl.ptr(scratch), nbytes)
    assert L.gdn_test_delta_wait_timeout(*args, 10, stream(), check=False) == gl.GDN_EINVAL   # limit below 1 us
    assert L.gdn_test_delta_wait_timeout(*args, 1_000_000, stream()) == gl.GDN_OK
    assert L.gdn_sync_status(stream(), check=False) == gl.GDN_ETIMEOUT
    assert "delta-rule" in L.last_error()
    assert L.gdn_sync_status(stream(), check=False) == gl.GDN_OK      # reading cleared the error word
    sout = torch.empty(spec.n_v_heads, spec.dv, spec.dk, dtype=torch.float32, device=DEV)
    o = torch.empty(n, spec.c_v, dtype=torch.float16, device=DEV)
    L.gdn_delta_rule(ctypes.byref(s), gl.ptr(qkv), gl.ptr(lad), gl.ptr(bd), n, 0, gl.ptr(sout), gl.ptr(o),
                     gl.ptr(scratch), nbytes, stream())
    sync(L)
    ro, rS = OL.gated_delta_rule(qe, ke, ve, la, b, np.zeros((spec.n_v_heads, spec.dv, spec.dk)))
    assert rel_l2(o.float().cpu().numpy(), ro.reshape(n, -1)) <= 2e-3
    assert rel_l2(sout.cpu().numpy(), rS) <= 2e-3


def test_delta_rule_state_aliasing(L):
    spec = DELTA_SPECS[1]
    _, dev, s = _layer(spec, L)
    rng = np.random.default_rng(77)
    n = 150
    qkv_h, qe, ke, ve, la, b = _delta_inputs(spec, n, rng)
    S0 = rng.normal(0, 0.3, size=(spec.n_v_heads, spec.dv, spec.dk)).astype(np.float32)
    qkv, lad, bd, st = f16_dev(qkv_h), f32_dev(la), f32_dev(b), f32_dev(S0)
    o = torch.empty(n, spec.c_v, dtype=torch.float16, device=DEV)
    nbytes = L.gdn_delta_rule_scratch_size(ctypes.byref(s), n)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    L.gdn_delta_rule(ctypes.byref(s), gl.ptr(qkv), gl.ptr(lad), gl.ptr(bd), n, gl.ptr(st), gl.ptr(st), gl.ptr(o),
                     gl.ptr(scratch), nbytes, stream())
    sync(L)
    ro, rS = OL.gated_delta_rule(qe, ke, ve, la, b, S0)
    assert rel_l2(st.cpu().numpy(), rS) <= 2e-3
    assert rel_l2(o.float().cpu().numpy(), ro.reshape(n, -1)) <= 2e-3


def test_delta_rule_reports_fp16_overflow(L):
    """A state whose fp16 operand image would overflow (|S| > 65504) is
    reported as GDN_ERANGE; the next call with a state in range is clean."""
    spec = DELTA_SPECS[1]
    _, dev, s = _layer(spec, L)
    rng = np.random.default_rng(78)
    n = 100
    qkv_h, qe, ke, ve, la, b = _delta_inputs(spec, n, rng)
    qkv, lad, bd = f16_dev(qkv_h), f32_dev(la), f32_dev(b)
    o = torch.empty(n, spec.c_v, dtype=torch.float16, device=DEV)
    nbytes = L.gdn_delta_rule_scratch_size(ctypes.byref(s), n)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    for scale, want in ((1.0e5, gl.GDN_ERANGE), (0.3, gl.GDN_OK)):
        st = f32_dev(rng.normal(0, scale, size=(spec.n_v_heads, spec.dv, spec.dk)))
        L.gdn_delta_rule(ctypes.byref(s), gl.ptr(qkv), gl.ptr(lad), gl.ptr(bd), n, gl.ptr(st), gl.ptr(st), gl.ptr(o),
                         gl.ptr(scratch), nbytes, stream())
        assert L.gdn_sync_status(stream(), check=False) == want


# ------------------------------------------------------------------ step 4

@pytest.mark.parametrize("spec", [synth.SPECS["tiny_f32"], synth.SPECS["h2560"], synth.SPECS["h1024"]],
                         ids=lambda s: s.name)
@pytest.mark.parametrize("n", [1, 7, 300])
def test_gated_norm_stage(L, spec, n):
    layer, dev, s = _layer(spec, L)
    rng = np.random.default_rng(n + 5)
    # o in fp16, as gdn_delta_rule writes it
    o = f16_round(rng.normal(0, 0.05, size=(n, spec.c_v)))
    zbits = synth._to_bf16_bits(rng.normal(0, 1, size=(n, spec.c_v)).astype(np.float32))
    z = synth.bf16_bits_to_f32(zbits)
    od, zd = f16_dev(o), bf16_dev(zbits)
    ref = OL.gated_rmsnorm(o.reshape(n, spec.n_v_heads, spec.dv), z.reshape(n, spec.n_v_heads, spec.dv),
                           layer["norm_w"], 1e-6).reshape(n, -1)
    if spec.wtype == "f32":
        out = torch.empty(n, spec.c_v, dtype=torch.float32, device=DEV)
        L.gdn_gated_norm(ctypes.byref(s), gl.ptr(od), gl.ptr(zd), spec.c_v, n, 0, 0, gl.ptr(out), stream())
        sync(L)
        assert rel_l2(out.cpu().numpy(), ref) < 1e-5
    else:
        codes = torch.empty(n, spec.c_v, dtype=torch.float16, device=DEV)
        sc = torch.empty(n, dtype=torch.float32, device=DEV)
        L.gdn_gated_norm(ctypes.byref(s), gl.ptr(od), gl.ptr(zd), spec.c_v, n, gl.ptr(codes), gl.ptr(sc), 0, stream())
        sync(L)
        rq, rs = quant.quant_rows_i8(ref.astype(np.float32))
        gq = f16_codes(codes)
        assert np.all(np.abs(gq - rq) <= 1)
        assert np.mean(gq != rq) < 1e-2
        assert rel_l2(sc.cpu().numpy(), rs) < 1e-5
