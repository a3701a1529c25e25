"""Helpers shared by the GPU tests: tensor conversions and oracle parameters."""
import numpy as np
import torch

from hybrid_gated_deltanet_q4k_gb300 import lib as gl
from hybrid_gated_deltanet_q4k_gb300 import synth
from oracle import q4k

DEV = "cuda"


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    """bf16 device tensor from uint16 bit patterns."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def bf16_host_f32(t: torch.Tensor) -> np.ndarray:
    """Exact float32 values of a bf16 device tensor."""
    bits = t.view(torch.int16).cpu().numpy().view(np.uint16)
    return synth.bf16_bits_to_f32(bits)


def f16_codes(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().astype(np.float32).astype(np.int64)


def f32_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(DEV)


def oracle_params(spec, layer: dict, eps=1e-6) -> dict:
    p = dict(wtype=spec.wtype, hidden=spec.hidden, n_qk_heads=spec.n_qk_heads, n_v_heads=spec.n_v_heads,
             dk=spec.dk, dv=spec.dv, conv_w=layer["conv_w"], A_log=layer["A_log"], dt_bias=layer["dt_bias"],
             norm_w=layer["norm_w"], eps_l2=eps, eps_rms=eps, q_scale=spec.dk ** -0.5)
    if spec.wtype == "q4k":
        p["w_in"] = q4k.pack_q4k(layer["w_in"])
        p["w_out"] = q4k.pack_q4k(layer["w_out"])
    else:
        p["w_in"], p["w_out"] = layer["w_in"], layer["w_out"]
    return p


def f16_round(x) -> np.ndarray:
    """Values rounded to IEEE fp16 (nearest even), returned as float32 (exact)."""
    return np.asarray(x).astype(np.float16).astype(np.float32)


def f16_dev(a: np.ndarray) -> torch.Tensor:
    """fp16 device tensor of the values (rounded to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a).astype(np.float16))).to(DEV)


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def stream() -> int:
    return gl.stream_handle()


def sync(L):
    assert L.gdn_sync_status(stream(), check=False) == gl.GDN_OK, L.last_error()


class Guarded:
    """A device buffer of n_bytes between two guard regions filled with a
    sentinel byte, so that any write outside the buffer shows up as a changed
    guard byte (the tests' substitute for a sanitizer).  The buffer starts
    4096 bytes into the allocation, so it keeps the allocation's alignment."""

    GUARD = 4096
    FILL = 0xA5

    def __init__(self, n_bytes: int, fill_inside: int | None = None):
        self.n = int(n_bytes)
        self.raw = torch.full((self.GUARD + self.n + self.GUARD,), self.FILL, dtype=torch.uint8, device=DEV)
        if fill_inside is not None:
            self.raw[self.GUARD:self.GUARD + self.n] = fill_inside

    def view(self, dtype: torch.dtype, shape) -> torch.Tensor:
        return self.raw[self.GUARD:self.GUARD + self.n].view(dtype).view(shape)

    def intact(self) -> bool:
        return bool((self.raw[:self.GUARD] == self.FILL).all().item()) and bool(
            (self.raw[self.GUARD + self.n:] == self.FILL).all().item())


def guarded(shape, dtype: torch.dtype, init: torch.Tensor | None = None):
    """(Guarded, view) for a tensor of this shape and dtype, optionally copied from init."""
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    g = Guarded(n)
    v = g.view(dtype, shape)
    if init is not None:
        v.copy_(init)
    else:
        v.zero_()
    return g, v
