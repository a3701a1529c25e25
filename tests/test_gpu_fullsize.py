"""Full-size parity: the 9B-like layer (hidden 4096, 16 q/k heads and 32 v heads
of 128) at N = 32768, in the single-pass launch configuration the benchmark
times.

gdn_prefill is run once; the same pipeline is then run stage by stage through
the stage entry points and must give the same bits.  The oracle checks what
it can compute at this size: the decoded weights in full, sampled rows of
every integer stage (bit-exact), sampled tokens of the conv and gated norm,
and the whole 32768-token recurrence of two value heads (relative L2 2e-3).
"""
import ctypes

import numpy as np
import pytest
import torch

from hybrid_gated_deltanet_q4k_gb300 import lib as gl
from hybrid_gated_deltanet_q4k_gb300 import synth
from hybrid_gated_deltanet_q4k_gb300.api import DeviceLayer
from oracle import layer as OL
from oracle import q4k, quant

from gpu_util import DEV, bf16_dev, bf16_host_f32, f16_codes, f32_dev, rel_l2, stream, sync

pytestmark = pytest.mark.gpu


def test_h4096_n32768_prefill():
    L = gl.load(build=True)
    spec = synth.SPECS["h4096"]
    n, H, hv, d = spec.n_tokens, spec.hidden, spec.n_v_heads, spec.dk
    c_qk, c_v, c_conv = spec.c_qk, spec.c_v, spec.c_conv
    nbf, r_in = 2 * c_qk + 2 * c_v, spec.r_in
    layer = synth.make_layer(spec)
    tok = synth.make_tokens(spec, n, seed=spec.seed + 10)
    dl = DeviceLayer(spec, layer)
    x = bf16_dev(tok["x_bits"])
    la, bb = f32_dev(tok["log_a"]), f32_dev(tok["b"])
    state, conv = dl.new_state()
    y = torch.empty(n, H, dtype=torch.bfloat16, device=DEV)
    ws = dl.new_workspace(n)
    dl.prefill(x, None, state, conv, y, ws, gate_log_a=la, gate_b=bb)
    sync(L)

    # the same pipeline, stage by stage
    s = dl.struct(la, bb)
    sp = ctypes.byref(s)
    st = stream()
    wc_in = torch.empty(r_in, H, dtype=torch.float16, device=DEV)
    ws_in = torch.empty(r_in, dtype=torch.float32, device=DEV)
    wc_out = torch.empty(H, c_v, dtype=torch.float16, device=DEV)
    ws_out = torch.empty(H, dtype=torch.float32, device=DEV)
    L.gdn_q4k_deq_codes(gl.ptr(dl.dev["w_in"]), r_in, H, gl.ptr(wc_in), gl.ptr(ws_in), st)
    L.gdn_q4k_deq_codes(gl.ptr(dl.dev["w_out"]), H, c_v, gl.ptr(wc_out), gl.ptr(ws_out), st)
    xc = torch.empty(n, H, dtype=torch.float16, device=DEV)
    sx = torch.empty(n, dtype=torch.float32, device=DEV)
    L.gdn_quant_rows(gl.ptr(x), n, H, gl.ptr(xc), gl.ptr(sx), st)
    qkvz = torch.empty(n, nbf, dtype=torch.bfloat16, device=DEV)
    ba = torch.empty(n, 2 * hv, dtype=torch.float32, device=DEV)
    L.gdn_gemm_codes(gl.ptr(xc), gl.ptr(sx), gl.ptr(wc_in), gl.ptr(ws_in), n, r_in, H, gl.ptr(qkvz), nbf, nbf,
                     gl.ptr(ba), 2 * hv, st)
    conv2 = torch.zeros(c_conv, 3, dtype=torch.float32, device=DEV)
    qkv = torch.empty(n, c_conv, dtype=torch.float16, device=DEV)
    L.gdn_conv(sp, gl.ptr(qkvz), nbf, n, gl.ptr(conv2), gl.ptr(ba), 2 * hv, gl.ptr(qkv), 0, 0, st)
    L.gdn_conv_state_update(sp, gl.ptr(qkvz), nbf, n, gl.ptr(conv2), st)
    nbytes = L.gdn_delta_rule_scratch_size(sp, n)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    state2 = torch.empty_like(state)
    o = torch.empty(n, c_v, dtype=torch.float16, device=DEV)
    L.gdn_delta_rule(sp, gl.ptr(qkv), gl.ptr(la), gl.ptr(bb), n, 0, gl.ptr(state2), gl.ptr(o), gl.ptr(scratch), nbytes, st)
    del scratch
    oc = torch.empty(n, c_v, dtype=torch.float16, device=DEV)
    so = torch.empty(n, dtype=torch.float32, device=DEV)
    z = qkvz[:, c_conv:]
    L.gdn_gated_norm(sp, gl.ptr(o), gl.ptr(z), nbf, n, gl.ptr(oc), gl.ptr(so), 0, st)
    y2 = torch.empty_like(y)
    L.gdn_gemm_codes(gl.ptr(oc), gl.ptr(so), gl.ptr(wc_out), gl.ptr(ws_out), n, H, c_v, gl.ptr(y2), H, H, 0, 0, st)
    sync(L)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(state, state2) and torch.equal(conv, conv2)

    rng = np.random.default_rng(0)
    rows = np.sort(np.concatenate([[0, 1, 2, 3, n - 1], rng.choice(n, 59, replace=False)]))
    # 1a: every decoded weight, bit-exact
    bin_ = dl.host_blocks["w_in"]
    rq_in, rs_in = quant.quant_rows_i8(q4k.unpack_q4k(bin_, r_in, H))
    assert np.array_equal(f16_codes(wc_in), rq_in.astype(np.int64))
    assert np.array_equal(ws_in.cpu().numpy().view(np.uint32), rs_in.view(np.uint32))
    rq_out, rs_out = quant.quant_rows_i8(q4k.unpack_q4k(dl.host_blocks["w_out"], H, c_v))
    assert np.array_equal(f16_codes(wc_out), rq_out.astype(np.int64))
    # 1b + 1c on sampled tokens, bit-exact
    rqx, rsx = quant.quant_rows_i8(tok["x"][rows])
    assert np.array_equal(f16_codes(xc[rows]), rqx.astype(np.int64))
    P = quant.gemm_q8(rqx, rsx, rq_in, rs_in)
    assert np.array_equal(bf16_host_f32(qkvz[rows]).view(np.uint32), quant.bf16_round(P[:, :nbf]).view(np.uint32))
    assert np.array_equal(ba[rows].cpu().numpy().view(np.uint32), P[:, nbf:].view(np.uint32))
    # 2: sampled tokens from the GPU's own projection
    p = dict(n_qk_heads=spec.n_qk_heads, n_v_heads=hv, dk=d, dv=d, conv_w=layer["conv_w"], eps_l2=1e-6,
             q_scale=d ** -0.5)
    raw_all = bf16_host_f32(qkvz[:, :c_conv])
    for t in rows[rows >= 3][:16]:
        qq, kk, vv, _ = OL.conv_stage(p, raw_all[t - 3:t + 1], np.zeros((c_conv, 3)))
        ref = np.concatenate([qq[-1].ravel(), kk[-1].ravel(), vv[-1].ravel()])
        got = qkv[t].cpu().numpy()
        assert np.all(np.abs(got - ref) <= (2 ** -11 + 3e-5) * np.abs(ref) + 1e-6 * np.abs(ref).max())
    # 3: the whole recurrence of two value heads from the GPU's own q, k, v
    qkv_h = qkv.cpu().numpy().astype(np.float64)
    for h in (0, hv - 1):
        hk = h // (hv // spec.n_qk_heads)
        qh = qkv_h[:, hk * d:(hk + 1) * d][:, None, :]
        kh = qkv_h[:, c_qk + hk * d:c_qk + (hk + 1) * d][:, None, :]
        vh = qkv_h[:, 2 * c_qk + h * d:2 * c_qk + (h + 1) * d][:, None, :]
        ro, rS = OL.gated_delta_rule(qh, kh, vh, tok["log_a"][:, h:h + 1], tok["b"][:, h:h + 1], np.zeros((1, d, d)))
        assert rel_l2(o[:, h * d:(h + 1) * d].float().cpu().numpy(), ro[:, 0]) <= 2e-3
        assert rel_l2(state[h].cpu().numpy(), rS[0]) <= 2e-3
    # 4: gated norm on sampled tokens
    o_s = o[rows].float().cpu().numpy().reshape(len(rows), hv, d)
    z_s = bf16_host_f32(qkvz[rows, c_conv:]).reshape(len(rows), hv, d)
    oh = OL.gated_rmsnorm(o_s, z_s, layer["norm_w"], 1e-6).reshape(len(rows), -1)
    rqo, rso = quant.quant_rows_i8(oh.astype(np.float32))
    gq = f16_codes(oc[rows])
    assert np.all(np.abs(gq - rqo) <= 1) and np.mean(gq != rqo) < 1e-2
    assert rel_l2(so[rows].cpu().numpy(), rso) < 1e-5
    # 5: output projection on sampled tokens from the GPU's own codes, bit-exact
    Y = quant.gemm_q8(gq, so[rows].cpu().numpy(), rq_out, rs_out)
    assert np.array_equal(bf16_host_f32(y[rows]).view(np.uint32), quant.bf16_round(Y).view(np.uint32))
