"""gdn_prefill_ckpt: recurrent-state and conv-state snapshots every K tokens.

Snapshot k must be, bit for bit, what gdn_prefill over the first (k+1)K tokens
leaves in state_out and conv_state (same chunks, same arithmetic), also when
the prompt runs in several workspace passes; resuming from a snapshot must
reproduce the rest of the full prefill bit for bit.
"""
import numpy as np
import pytest
import torch

from hybrid_gated_deltanet_q4k_gb300 import lib as gl
from hybrid_gated_deltanet_q4k_gb300 import synth
from hybrid_gated_deltanet_q4k_gb300.api import DeviceLayer

from oracle import layer as OL

from gpu_util import DEV, bf16_dev, bf16_host_f32, f32_dev, oracle_params, rel_l2, sync

pytestmark = pytest.mark.gpu

SMALL = synth.LayerSpec("small", 512, 2, 4, 128, 128, 0, "q4k", 11, "softplus_normal")


def _x(tok, a, b):
    return bf16_dev(tok["x_bits"][a:b])


def _prefill(dl, tok, a, b, state=None, conv=None, ws_tokens=None):
    if state is None:
        state, conv = dl.new_state()
    y = torch.empty(b - a, dl.spec.hidden, dtype=torch.bfloat16, device=DEV)
    dl.prefill(_x(tok, a, b), state, state, conv, y, dl.new_workspace(ws_tokens or (b - a)),
               gate_log_a=f32_dev(tok["log_a"][a:b]), gate_b=f32_dev(tok["b"][a:b]))
    return y, state, conv


@pytest.mark.parametrize("spec_name,n,every,ws_tokens", [("small", 1000, 256, None), ("small", 1000, 192, 320),
                                                          ("small", 5200, 1024, None), ("h2560", 4500, 2048, 1024)])
def test_snapshots_equal_prefix_prefills(spec_name, n, every, ws_tokens):
    spec = SMALL if spec_name == "small" else synth.SPECS[spec_name]
    layer = synth.make_layer(spec)
    tok = synth.make_tokens(spec, n, seed=n + every)
    dl = DeviceLayer(spec, layer)
    k = n // every
    cs = torch.full((k, spec.n_v_heads, spec.dv, spec.dk), float("nan"), device=DEV)
    cc = torch.full((k, spec.c_conv, 3), float("nan"), device=DEV)
    state, conv = dl.new_state()
    y = torch.empty(n, spec.hidden, dtype=torch.bfloat16, device=DEV)
    dl.prefill_ckpt(_x(tok, 0, n), None, state, conv, y, dl.new_workspace(ws_tokens or n), every, cs, cc,
                    gate_log_a=f32_dev(tok["log_a"]), gate_b=f32_dev(tok["b"]))
    sync(dl.lib)
    yf, sf, cf = _prefill(dl, tok, 0, n)
    sync(dl.lib)
    assert torch.equal(y.view(torch.int16), yf.view(torch.int16))
    assert torch.equal(state, sf) and torch.equal(conv, cf)
    for j in range(k):
        p = (j + 1) * every
        _, sp, cp = _prefill(dl, tok, 0, p)
        sync(dl.lib)
        assert torch.equal(cs[j], sp), j
        assert torch.equal(cc[j], cp), j
    # resume from the last snapshot: the rest equals the full prefill's tail
    p = k * every
    if p < n:
        yr, sr, cr = _prefill(dl, tok, p, n, state=cs[k - 1].clone(), conv=cc[k - 1].clone())
        sync(dl.lib)
        assert torch.equal(yr.view(torch.int16), yf[p:].view(torch.int16))
        assert torch.equal(sr, sf) and torch.equal(cr, cf)


@pytest.mark.parametrize("n,every", [(700, 256), (1000, 192)])
def test_oracle_resumed_from_a_snapshot_continues_the_prompt(n, every):
    """A GPU snapshot handed to the oracle: the oracle, started from snapshot k
    (its state and conv tail, fp32 values taken exactly), runs the rest of the
    prompt, and its outputs and final state agree with the GPU's full prefill
    within the end-to-end tolerances (y 1e-2 through the int8 projections, the
    state 2e-3 of the recurrence).  So a snapshot is a state the method can
    resume from, not only a copy of the GPU's own prefix prefill."""
    spec = SMALL
    layer = synth.make_layer(spec)
    tok = synth.make_tokens(spec, n, seed=n + 7 * every)
    dl = DeviceLayer(spec, layer)
    k = n // every
    cs = torch.empty(k, spec.n_v_heads, spec.dv, spec.dk, device=DEV)
    cc = torch.empty(k, spec.c_conv, 3, device=DEV)
    state, conv = dl.new_state()
    y = torch.empty(n, spec.hidden, dtype=torch.bfloat16, device=DEV)
    dl.prefill_ckpt(_x(tok, 0, n), None, state, conv, y, dl.new_workspace(n), every, cs, cc,
                    gate_log_a=f32_dev(tok["log_a"]), gate_b=f32_dev(tok["b"]))
    sync(dl.lib)
    p = oracle_params(spec, layer)
    yh = bf16_host_f32(y)
    for j in (0, k - 1):
        t0 = (j + 1) * every
        ref = OL.layer_forward(p, tok["x"][t0:], S0=cs[j].cpu().numpy().astype(np.float64),
                               conv_tail=cc[j].cpu().numpy().astype(np.float64),
                               gate_log_a=tok["log_a"][t0:], gate_b=tok["b"][t0:])
        assert rel_l2(yh[t0:], ref["y"]) <= 1e-2, j
        assert rel_l2(state.cpu().numpy(), ref["state"]) <= 2e-3, j
        assert np.array_equal(conv.cpu().numpy(), ref["conv_tail"].astype(np.float32)), j


def test_ckpt_argument_checks():
    spec = SMALL
    dl = DeviceLayer(spec, synth.make_layer(spec))
    tok = synth.make_tokens(spec, 300, seed=3)
    state, conv = dl.new_state()
    y = torch.empty(300, spec.hidden, dtype=torch.bfloat16, device=DEV)
    ws = dl.new_workspace(300)
    cs = torch.empty(4, spec.n_v_heads, spec.dv, spec.dk, device=DEV)
    cc = torch.empty(4, spec.c_conv, 3, device=DEV)
    for every in (0, 100, -64):
        assert dl.prefill_ckpt(_x(tok, 0, 300), None, state, conv, y, ws, every, cs, cc, check=False) == gl.GDN_EINVAL
    assert dl.prefill_ckpt(_x(tok, 0, 300), None, state, conv, y, ws, 64, None, cc, check=False) == gl.GDN_EINVAL
    # fewer tokens than one interval: no snapshot, no buffer needed
    assert dl.prefill_ckpt(_x(tok, 0, 300), None, state, conv, y, ws, 512, None, None, check=False) == gl.GDN_OK
    # a workspace of fewer than 64 tokens with snapshots
    small = dl.new_workspace(40)
    assert dl.prefill_ckpt(_x(tok, 0, 300), None, state, conv, y, small, 64, cs, cc, check=False) == gl.GDN_ENOMEM
    sync(dl.lib)
