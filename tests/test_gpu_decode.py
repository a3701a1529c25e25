"""The decode step (gdn_decode): one token per sequence, states and conv tails
updated in place.

* Its projection (int8 activation rows against the exactly decoded Q4_K /
  Q6_K weights, integer dot products per sub-block, fp32 sums) matches the
  oracle's exact product within fp32 rounding (relative L2 1e-6 on fp32
  outputs, one bf16 rounding on bf16 outputs), for any number of tokens
  (several launches past 8).
* One step on sequences with saved states matches the oracle's layer on that
  token with the same projections (y within 1e-2 relative L2, the
  int8-projection tolerance; the state within 2e-3, the recurrence tolerance;
  the conv tail exactly).
* A prefill followed by tokens decoded one at a time matches the oracle doing
  the same, and a batch of sequences decodes bit for bit as each sequence
  alone.
"""
import numpy as np
import pytest
import torch

from hybrid_gated_deltanet_q4k_gb300 import lib as gl
from hybrid_gated_deltanet_q4k_gb300 import synth
from hybrid_gated_deltanet_q4k_gb300.api import DeviceLayer
from oracle import layer as OL
from oracle import q4k, q6k, quant

from gpu_util import DEV, bf16_dev, bf16_host_f32, f32_dev, oracle_params, rel_l2, stream, sync

pytestmark = pytest.mark.gpu

SMALL = synth.LayerSpec("small", 512, 2, 4, 128, 128, 0, "q4k", 11, "softplus_normal")


@pytest.fixture(scope="module")
def L():
    return gl.load(build=True)


@pytest.mark.parametrize("fmt,rows,cols,n,n_bf16", [("q4k", 300, 1024, 1, 300), ("q4k", 1000, 4096, 8, 700),
                                                     ("q6k", 517, 2048, 9, 0), ("q6k", 64, 16384, 3, 40),
                                                     ("q4k", 12352, 4096, 1, 12288),
                                                     # one token, an odd row count: the last row pair has one row,
                                                     # and rows 150 / 151 of a pair go to the bf16 / fp32 outputs
                                                     ("q4k", 301, 1024, 1, 151),
                                                     # 2 tokens, and 6 tokens computed as 8 (two zero rows)
                                                     ("q4k", 200, 512, 2, 100), ("q6k", 300, 1024, 6, 150)])
def test_decode_gemv_matches_oracle(L, fmt, rows, cols, n, n_bf16):
    rng = np.random.default_rng(rows + cols + n)
    w = rng.normal(0, 0.02, size=(rows, cols)).astype(np.float32)
    w[0] = 0.0
    blocks = (q6k.pack_q6k if fmt == "q6k" else q4k.pack_q4k)(w)
    wf = (q6k.unpack_q6k if fmt == "q6k" else q4k.unpack_q4k)(blocks, rows, cols)
    x = (rng.normal(0, 1, size=(n, cols)) * 10.0 ** rng.uniform(-2, 2, size=(n, 1))).astype(np.float32)
    qx, sx = quant.quant_rows_i8(x)
    ref = quant.matvec_exact_weights(qx, sx, wf)               # fp64 [n][rows]
    xc = torch.from_numpy(qx.astype(np.float16)).to(DEV)
    sxd = f32_dev(sx)
    b = torch.from_numpy(blocks).to(DEV)
    ob = torch.zeros(n, max(n_bf16, 1), dtype=torch.int16, device=DEV)
    of = torch.zeros(n, max(rows - n_bf16, 1), dtype=torch.float32, device=DEV)
    L.gdn_decode_gemv(gl.ptr(b), int(fmt == "q6k"), rows, cols, gl.ptr(xc), gl.ptr(sxd), n, gl.ptr(ob), ob.shape[1],
                      n_bf16, gl.ptr(of), of.shape[1], stream())
    sync(L)
    if n_bf16:
        # one bf16 rounding of an fp32 value within ~1e-6 of the exact sum: at most one bf16 step apart
        got = synth.bf16_bits_to_f32(ob.cpu().numpy().view(np.uint16)[:, :n_bf16]).astype(np.float64)
        want = ref[:, :n_bf16]
        assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-6 * np.abs(want).max())
        assert rel_l2(got, want) <= 2.0 ** -8
    if rows > n_bf16:
        got = of.cpu().numpy()[:, : rows - n_bf16]
        assert rel_l2(got, ref[:, n_bf16:]) <= 1e-6


def _tail_close(got, want):
    """Conv tails of decoded tokens: raw projection outputs rounded to bf16 from
    an fp32 (GPU) or fp64 (oracle) sum can straddle a rounding boundary: one
    bf16 step at most."""
    want = np.asarray(want, np.float64)
    return np.all(np.abs(np.asarray(got, np.float64) - want) <= 2.0 ** -7 * np.abs(want) + 1e-30)


def _saved_states(spec, n, seed):
    rng = np.random.default_rng(seed)
    st = (0.05 * rng.standard_normal((n, spec.n_v_heads, spec.dv, spec.dk))).astype(np.float32)
    cv = rng.standard_normal((n, spec.c_conv, 3)).astype(np.float32)
    if spec.wtype == "q4k":        # the conv tail holds raw bf16 projection outputs
        cv = synth.bf16_bits_to_f32(synth._to_bf16_bits(cv))
    return st, cv


@pytest.mark.parametrize("name,n,gates,q6", [("small", 1, True, ()), ("small", 5, False, ()),
                                              ("small", 11, True, ("w_out",)), ("small", 1, False, ("w_in", "w_out")),
                                              ("h2560", 3, True, ()), ("h2560", 1, True, ()),
                                              ("tiny_f32", 4, True, ())])
def test_decode_step_matches_oracle(name, n, gates, q6):
    spec = SMALL if name == "small" else synth.SPECS[name]
    layer = synth.make_layer(spec)
    tok = synth.make_tokens(spec, n, seed=n + 60)
    dl = DeviceLayer(spec, layer, q6k=q6)
    st0, cv0 = _saved_states(spec, n, seed=n)
    state, conv = torch.from_numpy(st0).to(DEV), torch.from_numpy(cv0).to(DEV)
    q4 = spec.wtype == "q4k"
    x = bf16_dev(tok["x_bits"]) if q4 else f32_dev(tok["x"])
    y = torch.empty(n, spec.hidden, dtype=torch.bfloat16 if q4 else torch.float32, device=DEV)
    ws = dl.new_decode_workspace(n)
    la, bb = (f32_dev(tok["log_a"]), f32_dev(tok["b"])) if gates else (None, None)
    dl.decode(x, state, conv, y, ws, gate_log_a=la, gate_b=bb)
    sync(dl.lib)
    p = oracle_params(spec, layer)
    from oracle import q6k as O6
    for nm in q6:
        p[nm], p[nm + "_fmt"] = O6.pack_q6k(layer[nm]), "q6k"
    yh = bf16_host_f32(y) if q4 else y.cpu().numpy()
    for s in range(n):
        ref = OL.layer_forward(p, tok["x"][s:s + 1], S0=st0[s].astype(np.float64), conv_tail=cv0[s],
                               gate_log_a=tok["log_a"][s:s + 1] if gates else None,
                               gate_b=tok["b"][s:s + 1] if gates else None, decode=True)
        assert rel_l2(yh[s:s + 1], ref["y"]) <= 1e-2, s
        assert rel_l2(state[s].cpu().numpy(), ref["state"]) <= 2e-3, s
        if q4:
            c = conv[s].cpu().numpy()
            assert np.array_equal(c[:, :2], cv0[s][:, 1:]), s          # the older inputs move up, exactly
            assert _tail_close(c[:, 2], ref["conv_tail"][:, 2]), s


def test_prefill_then_decode_matches_oracle_prefill():
    """Prefill 200 tokens, then decode 40 more one at a time on the same state
    and conv tail: against the oracle doing the same (its prefill of the 200,
    then its decode step per token), and within the recurrence tolerance of
    the oracle's prefill of all 240."""
    spec = SMALL
    layer = synth.make_layer(spec)
    n0, m = 200, 40
    tok = synth.make_tokens(spec, n0 + m, seed=77)
    dl = DeviceLayer(spec, layer)
    state, conv = dl.new_state()
    y0 = torch.empty(n0, spec.hidden, dtype=torch.bfloat16, device=DEV)
    dl.prefill(bf16_dev(tok["x_bits"][:n0]), None, state, conv, y0, dl.new_workspace(n0),
               gate_log_a=f32_dev(tok["log_a"][:n0]), gate_b=f32_dev(tok["b"][:n0]))
    ws = dl.new_decode_workspace(1)
    ys = []
    st1, cv1 = state[None], conv[None]          # views: [1][...] of the same buffers
    for t in range(n0, n0 + m):
        y = torch.empty(1, spec.hidden, dtype=torch.bfloat16, device=DEV)
        dl.decode(bf16_dev(tok["x_bits"][t:t + 1]), st1, cv1, y, ws, gate_log_a=f32_dev(tok["log_a"][t:t + 1]),
                  gate_b=f32_dev(tok["b"][t:t + 1]))
        ys.append(y)
    sync(dl.lib)
    p = oracle_params(spec, layer)
    r0 = OL.layer_forward(p, tok["x"][:n0], gate_log_a=tok["log_a"][:n0], gate_b=tok["b"][:n0])
    S, tail, yr = r0["state"], r0["conv_tail"], []
    for t in range(n0, n0 + m):
        r = OL.layer_forward(p, tok["x"][t:t + 1], S0=S, conv_tail=tail, gate_log_a=tok["log_a"][t:t + 1],
                             gate_b=tok["b"][t:t + 1], decode=True)
        S, tail = r["state"], r["conv_tail"]
        yr.append(r["y"])
    yd = bf16_host_f32(torch.cat(ys))
    assert rel_l2(yd, np.concatenate(yr)) <= 1e-2
    assert rel_l2(state.cpu().numpy(), S) <= 2e-3
    assert _tail_close(conv.cpu().numpy(), tail)
    # against the oracle's prefill of all 240 tokens: the decode projections use
    # the exact weights where the prefill's use int8 weight rows (a half step
    # of the row scale per weight), which moves this state by about 1%
    full = OL.layer_forward(p, tok["x"], gate_log_a=tok["log_a"], gate_b=tok["b"])
    assert rel_l2(state.cpu().numpy(), full["state"]) <= 3e-2


@pytest.mark.parametrize("q6", [(), ("w_in", "w_out")])
def test_decode_batch_equals_each_sequence_alone(q6):
    """One sequence alone takes the one-token projection kernels; 13 take two
    launches of the batched ones (8 + 5 tokens).  Every sequence's results are
    the same bits, for Q4_K and for Q6_K projections."""
    spec = synth.SPECS["h2560"]
    layer = synth.make_layer(spec)
    n = 13
    tok = synth.make_tokens(spec, n, seed=5)
    dl = DeviceLayer(spec, layer, q6k=q6)
    st0, cv0 = _saved_states(spec, n, seed=9)
    sb, cb = torch.from_numpy(st0).to(DEV), torch.from_numpy(cv0).to(DEV)
    yb = torch.empty(n, spec.hidden, dtype=torch.bfloat16, device=DEV)
    dl.decode(bf16_dev(tok["x_bits"]), sb, cb, yb, dl.new_decode_workspace(n), gate_log_a=f32_dev(tok["log_a"]),
              gate_b=f32_dev(tok["b"]))
    ws1 = dl.new_decode_workspace(1)
    for s in range(n):
        ss, cs = torch.from_numpy(st0[s:s + 1]).to(DEV), torch.from_numpy(cv0[s:s + 1]).to(DEV)
        ys = torch.empty(1, spec.hidden, dtype=torch.bfloat16, device=DEV)
        dl.decode(bf16_dev(tok["x_bits"][s:s + 1]), ss, cs, ys, ws1, gate_log_a=f32_dev(tok["log_a"][s:s + 1]),
                  gate_b=f32_dev(tok["b"][s:s + 1]))
        sync(dl.lib)
        assert torch.equal(ys.view(torch.int16), yb[s:s + 1].view(torch.int16)), s
        assert torch.equal(ss[0], sb[s]) and torch.equal(cs[0], cb[s]), s


def test_decode_argument_checks(L):
    spec = SMALL
    dl = DeviceLayer(spec, synth.make_layer(spec))
    st, cv = dl.new_batch_state(2)
    x = torch.zeros(2, spec.hidden, dtype=torch.bfloat16, device=DEV)
    y = torch.empty_like(x)
    ws = dl.new_decode_workspace(2)
    assert dl.decode(x, st, cv, y, ws[:256], check=False) == gl.GDN_ENOMEM
    assert dl.decode_workspace_bytes(gl.GDN_MAX_SEQS + 1) == 0
    s = dl.struct()
    import ctypes
    assert L.gdn_decode(ctypes.byref(s), gl.ptr(x), 0, gl.ptr(st), gl.ptr(cv), gl.ptr(y), gl.ptr(ws), ws.numel(),
                        stream(), check=False) == gl.GDN_EINVAL


def test_decode_at_the_maximum_number_of_sequences():
    """GDN_MAX_SEQS sequences in one call (32 launches of the 8-token
    projection kernels): sampled sequences, the last included, against the
    oracle's decode step."""
    spec = SMALL
    layer = synth.make_layer(spec)
    n = gl.GDN_MAX_SEQS
    tok = synth.make_tokens(spec, n, seed=77)
    dl = DeviceLayer(spec, layer)
    st0, cv0 = _saved_states(spec, n, seed=78)
    state, conv = torch.from_numpy(st0).to(DEV), torch.from_numpy(cv0).to(DEV)
    y = torch.empty(n, spec.hidden, dtype=torch.bfloat16, device=DEV)
    dl.decode(bf16_dev(tok["x_bits"]), state, conv, y, dl.new_decode_workspace(n), gate_log_a=f32_dev(tok["log_a"]),
              gate_b=f32_dev(tok["b"]))
    sync(dl.lib)
    p = oracle_params(spec, layer)
    yh = bf16_host_f32(y)
    for s in (0, 1, 7, 8, 129, n - 1):
        ref = OL.layer_forward(p, tok["x"][s:s + 1], S0=st0[s].astype(np.float64), conv_tail=cv0[s],
                               gate_log_a=tok["log_a"][s:s + 1], gate_b=tok["b"][s:s + 1], decode=True)
        assert rel_l2(yh[s:s + 1], ref["y"]) <= 1e-2, s
        assert rel_l2(state[s].cpu().numpy(), ref["state"]) <= 2e-3, s
        c = conv[s].cpu().numpy()
        assert np.array_equal(c[:, :2], cv0[s][:, 1:]), s
        assert _tail_close(c[:, 2], ref["conv_tail"][:, 2]), s


@pytest.mark.parametrize("fmt", ["q4k", "q6k"])
def test_decode_gemv_token_result_independent_of_the_batch(L, fmt):
    """21 tokens in one call (launches of 16 + 5 tokens, or 8 + 8 + 5) give,
    bit for bit, what each token gives alone."""
    rng = np.random.default_rng(21)
    rows, cols, n = 500, 2048, 21
    w = rng.normal(0, 0.02, size=(rows, cols)).astype(np.float32)
    blocks = (q6k.pack_q6k if fmt == "q6k" else q4k.pack_q4k)(w)
    x = (rng.normal(0, 1, size=(n, cols)) * 10.0 ** rng.uniform(-2, 2, size=(n, 1))).astype(np.float32)
    qx, sx = quant.quant_rows_i8(x)
    xc = torch.from_numpy(qx.astype(np.float16)).to(DEV)
    sxd = f32_dev(sx)
    b = torch.from_numpy(blocks).to(DEV)
    ob = torch.zeros(1, dtype=torch.int16, device=DEV)

    def run(t0, t1):
        of = torch.zeros(t1 - t0, rows, dtype=torch.float32, device=DEV)
        L.gdn_decode_gemv(gl.ptr(b), int(fmt == "q6k"), rows, cols, gl.ptr(xc[t0:t1]), gl.ptr(sxd[t0:t1]), t1 - t0,
                          gl.ptr(ob), 1, 0, gl.ptr(of), rows, stream())
        sync(L)
        return of

    together = run(0, n)
    for t in range(n):
        assert torch.equal(run(t, t + 1)[0], together[t]), t
