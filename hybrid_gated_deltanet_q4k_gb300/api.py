"""User-facing wrapper: a GDN layer resident on the GPU, prefilled through the C ABI.

Weights are encoded to Q4_K on the host by the library's ``q4k_pack`` (or kept
fp32 for an F32 layer) and uploaded once; ``prefill`` enqueues one
``gdn_prefill`` call.  PyTorch only provides device memory and the stream.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import lib as gl


def pack_q4k(w: np.ndarray) -> np.ndarray:
    """Host Q4_K encoding through the library (``q4k_pack``)."""
    w = np.ascontiguousarray(w, np.float32)
    out = np.zeros((w.shape[0], w.shape[1] // 256 * 144), np.uint8)
    gl.load().q4k_pack(gl.ptr(w), w.shape[0], w.shape[1], gl.ptr(out))
    return out


def pack_q6k(w: np.ndarray) -> np.ndarray:
    """Host Q6_K encoding through the library (``q6k_pack``)."""
    w = np.ascontiguousarray(w, np.float32)
    out = np.zeros((w.shape[0], w.shape[1] // 256 * 210), np.uint8)
    gl.load().q6k_pack(gl.ptr(w), w.shape[0], w.shape[1], gl.ptr(out))
    return out


class DeviceLayer:
    """One GDN layer's parameters in device memory, in the layouts ``gdn_layer`` names."""

    def __init__(self, spec, params: dict, device: str = "cuda", eps_l2: float = 1e-6, eps_rms: float = 1e-6,
                 q_scale: float | None = None, blocks: dict | None = None, q6k: tuple = (), debug: bool = False):
        """q6k: names of the matrices ("w_in", "w_out") to hold in Q6_K instead of Q4_K.
        debug: run on the library's debug variant (index-checked kernels)."""
        self.spec = spec
        self.device = device
        self.lib = gl.load(debug=debug)
        self.q6k_mask = (1 if "w_in" in q6k else 0) | (2 if "w_out" in q6k else 0)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)  # noqa: E731
        if spec.wtype == "q4k":
            enc = {k: (pack_q6k if k in q6k else pack_q4k) for k in ("w_in", "w_out")}
            b_in = blocks["w_in"] if blocks else enc["w_in"](params["w_in"])
            b_out = blocks["w_out"] if blocks else enc["w_out"](params["w_out"])
            self.host_blocks = {"w_in": b_in, "w_out": b_out}
            self.dev = {"w_in": t(b_in), "w_out": t(b_out)}
        else:
            self.dev = {"w_in": t(params["w_in"].astype(np.float32)), "w_out": t(params["w_out"].astype(np.float32))}
        for k in ("conv_w", "A_log", "dt_bias", "norm_w"):
            self.dev[k] = t(params[k].astype(np.float32))
        self.eps_l2, self.eps_rms = eps_l2, eps_rms
        self.q_scale = spec.dk ** -0.5 if q_scale is None else q_scale

    def struct(self, gate_log_a=None, gate_b=None) -> gl.GdnLayer:
        L = gl.make_layer_struct(self.spec, self.dev, self.eps_l2, self.eps_rms, self.q_scale, gate_log_a, gate_b)
        L.q6k_mask = self.q6k_mask
        return L

    def workspace_bytes(self, ubatch_tokens: int) -> int:
        s = self.struct()
        return self.lib.gdn_workspace_size(ctypes.byref(s), int(ubatch_tokens))

    def new_workspace(self, ubatch_tokens: int) -> torch.Tensor:
        return torch.empty(self.workspace_bytes(ubatch_tokens), dtype=torch.uint8, device=self.device)

    def new_state(self) -> tuple:
        sp = self.spec
        state = torch.zeros(sp.n_v_heads, sp.dv, sp.dk, dtype=torch.float32, device=self.device)
        conv = torch.zeros(sp.c_conv, 3, dtype=torch.float32, device=self.device)
        return state, conv

    def prefill(self, x: torch.Tensor, state_in, state_out, conv_state, y, workspace, gate_log_a=None, gate_b=None,
                stream=None, check=True) -> int:
        """Enqueue gdn_prefill over x's rows; returns the status (raises if check and it is not 0)."""
        s = self.struct(gate_log_a, gate_b)
        return self.lib.gdn_prefill(ctypes.byref(s), gl.ptr(x), x.shape[0], gl.ptr(state_in), gl.ptr(state_out),
                                    gl.ptr(conv_state), gl.ptr(y), gl.ptr(workspace), workspace.numel(),
                                    gl.stream_handle(stream), check=check)

    def host_workspace_bytes(self, pass_tokens: int, gates: bool = False) -> int:
        """Device workspace of ``prefill_host`` for passes of ``pass_tokens`` (with or without drawn gates)."""
        s = self.struct()
        if gates:                   # only whether gates are drawn matters for the size
            s.gate_log_a = s.gate_b = 16
        return self.lib.gdn_host_workspace_size(ctypes.byref(s), int(pass_tokens))

    def new_host_workspace(self, pass_tokens: int, gates: bool = False) -> torch.Tensor:
        return torch.empty(self.host_workspace_bytes(pass_tokens, gates), dtype=torch.uint8, device=self.device)

    def prefill_host(self, x_host: torch.Tensor, state_in, state_out, conv_state, y_host: torch.Tensor, workspace,
                     pass_tokens: int = 0, gate_log_a=None, gate_b=None, stream=None, check=True) -> int:
        """Enqueue gdn_prefill_host: x_host, y_host (and the gates, if given) are pinned host tensors."""
        s = self.struct(gate_log_a, gate_b)
        return self.lib.gdn_prefill_host(ctypes.byref(s), gl.ptr(x_host), x_host.shape[0], gl.ptr(state_in),
                                         gl.ptr(state_out), gl.ptr(conv_state), gl.ptr(y_host), int(pass_tokens),
                                         gl.ptr(workspace), workspace.numel(), gl.stream_handle(stream), check=check)

    def batch_workspace_bytes(self, n_tokens: int, n_seqs: int) -> int:
        s = self.struct()
        return self.lib.gdn_batch_workspace_size(ctypes.byref(s), int(n_tokens), int(n_seqs))

    def new_batch_workspace(self, n_tokens: int, n_seqs: int) -> torch.Tensor:
        return torch.empty(self.batch_workspace_bytes(n_tokens, n_seqs), dtype=torch.uint8, device=self.device)

    def new_batch_state(self, n_seqs: int) -> tuple:
        sp = self.spec
        state = torch.zeros(n_seqs, sp.n_v_heads, sp.dv, sp.dk, dtype=torch.float32, device=self.device)
        conv = torch.zeros(n_seqs, sp.c_conv, 3, dtype=torch.float32, device=self.device)
        return state, conv

    def prefill_batch(self, x: torch.Tensor, cu_seqlens, state_in, state_out, conv_state, y, workspace,
                      gate_log_a=None, gate_b=None, stream=None, check=True) -> int:
        """Enqueue gdn_prefill_batch: x holds the sequences' tokens back to back, cu_seqlens (host, n_seqs + 1)
        their offsets; states [n_seqs][Hv][dv][dk] and conv tails [n_seqs][C_conv][3] are per sequence."""
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        s = self.struct(gate_log_a, gate_b)
        return self.lib.gdn_prefill_batch(ctypes.byref(s), gl.ptr(x), gl.ptr(cu), len(cu) - 1, gl.ptr(state_in),
                                          gl.ptr(state_out), gl.ptr(conv_state), gl.ptr(y), gl.ptr(workspace),
                                          workspace.numel(), gl.stream_handle(stream), check=check)

    def decode_workspace_bytes(self, n_seqs: int) -> int:
        s = self.struct()
        return self.lib.gdn_decode_workspace_size(ctypes.byref(s), int(n_seqs))

    def new_decode_workspace(self, n_seqs: int) -> torch.Tensor:
        return torch.empty(self.decode_workspace_bytes(n_seqs), dtype=torch.uint8, device=self.device)

    def decode(self, x: torch.Tensor, state, conv_state, y, workspace, gate_log_a=None, gate_b=None, stream=None,
               check=True) -> int:
        """Enqueue gdn_decode: one token per sequence (x [n_seqs][H]), states [n_seqs][Hv][dv][dk] and
        conv tails [n_seqs][C_conv][3] updated in place."""
        s = self.struct(gate_log_a, gate_b)
        return self.lib.gdn_decode(ctypes.byref(s), gl.ptr(x), x.shape[0], gl.ptr(state), gl.ptr(conv_state),
                                   gl.ptr(y), gl.ptr(workspace), workspace.numel(), gl.stream_handle(stream),
                                   check=check)

    def prefill_ckpt(self, x: torch.Tensor, state_in, state_out, conv_state, y, workspace, ckpt_every: int,
                     ckpt_state, ckpt_conv, gate_log_a=None, gate_b=None, stream=None, check=True) -> int:
        """Enqueue gdn_prefill_ckpt: as prefill, plus snapshots of the state [N // every][Hv][dv][dk] and conv
        state [N // every][C_conv][3] every ckpt_every tokens."""
        s = self.struct(gate_log_a, gate_b)
        return self.lib.gdn_prefill_ckpt(ctypes.byref(s), gl.ptr(x), x.shape[0], gl.ptr(state_in), gl.ptr(state_out),
                                         gl.ptr(conv_state), gl.ptr(y), int(ckpt_every), gl.ptr(ckpt_state),
                                         gl.ptr(ckpt_conv), gl.ptr(workspace), workspace.numel(),
                                         gl.stream_handle(stream), check=check)
