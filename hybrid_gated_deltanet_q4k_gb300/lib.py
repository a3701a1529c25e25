"""ctypes binding of ``libgdn`` (the C ABI declared in ``include/gdn.h``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Device buffers are passed as raw addresses (``int``); a helper turns
torch tensors into addresses.  Loading fails loudly if the library has not been
built: there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
import re

from . import build as _build

c_int32, c_int64, c_float, c_void_p, c_size_t = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t

GDN_OK, GDN_EINVAL, GDN_ENOMEM, GDN_ECUDA, GDN_ETIMEOUT, GDN_ERANGE, GDN_EINDEX = 0, -1, -2, -3, -4, -5, -6
GDN_W_Q4K, GDN_W_F32 = 0, 1
GDN_CHUNK = 64
GDN_MAX_SEQS = 256
GDN_N_STAGE_EVENTS = 8
GDN_NOALLOC_SCRATCH_BYTES = 48 << 20
STAGE_NAMES = ["dequant", "act_quant", "in_proj", "conv", "delta_rule", "gated_norm", "out_proj"]


class GdnLayer(ctypes.Structure):
    """Mirror of ``struct gdn_layer``."""
    _fields_ = [
        ("hidden", c_int32), ("n_qk_heads", c_int32), ("n_v_heads", c_int32), ("dk", c_int32), ("dv", c_int32),
        ("conv_taps", c_int32), ("wtype", c_int32), ("q6k_mask", c_int32),
        ("w_in", c_void_p), ("w_out", c_void_p), ("conv_w", c_void_p), ("A_log", c_void_p), ("dt_bias", c_void_p),
        ("norm_w", c_void_p), ("gate_log_a", c_void_p), ("gate_b", c_void_p),
        ("eps_l2", c_float), ("eps_rms", c_float), ("q_scale", c_float), ("reserved1", c_float),
    ]


_P = c_void_p
_SIGNATURES = {
    "q4k_pack": (c_int32, [_P, c_int64, c_int64, _P]),
    "q4k_deq_i8": (c_int32, [_P, c_int64, c_int64, _P, _P, _P]),
    "q6k_pack": (c_int32, [_P, c_int64, c_int64, _P]),
    "q6k_deq_i8": (c_int32, [_P, c_int64, c_int64, _P, _P, _P]),
    "gdn_q6k_deq_codes": (c_int32, [_P, c_int64, c_int64, _P, _P, _P]),
    "gdn_workspace_size": (c_size_t, [_P, c_int64]),
    "gdn_prefill": (c_int32, [_P, _P, c_int64, _P, _P, _P, _P, _P, c_size_t, _P]),
    "gdn_batch_workspace_size": (c_size_t, [_P, c_int64, c_int32]),
    "gdn_prefill_batch": (c_int32, [_P, _P, _P, c_int32, _P, _P, _P, _P, _P, c_size_t, _P]),
    "gdn_decode_workspace_size": (c_size_t, [_P, c_int32]),
    "gdn_decode": (c_int32, [_P, _P, c_int32, _P, _P, _P, _P, c_size_t, _P]),
    "gdn_decode_gemv": (c_int32, [_P, c_int32, c_int64, c_int64, _P, _P, c_int64, _P, c_int64, c_int64, _P, c_int64, _P]),
    "gdn_host_workspace_size": (c_size_t, [_P, c_int64]),
    "gdn_prefill_host": (c_int32, [_P, _P, c_int64, _P, _P, _P, _P, c_int64, _P, c_size_t, _P]),
    "gdn_prefill_ckpt": (c_int32, [_P, _P, c_int64, _P, _P, _P, _P, c_int64, _P, _P, _P, c_size_t, _P]),
    "gdn_attn_workspace_size": (c_size_t, [c_int64, c_int32, c_int32]),
    "gdn_attn_prefill": (c_int32, [_P, _P, _P, c_int64, c_int64, c_int32, c_int32, c_int32, c_float, _P, _P, c_size_t, _P]),
    "gdn_sync_status": (c_int32, [_P]),
    "gdn_last_error": (ctypes.c_char_p, []),
    "gdn_set_stage_events": (c_int32, [ctypes.POINTER(c_void_p), c_int32]),
    "gdn_q4k_deq_codes": (c_int32, [_P, c_int64, c_int64, _P, _P, _P]),
    "gdn_quant_rows": (c_int32, [_P, c_int64, c_int64, _P, _P, _P]),
    "gdn_gemm_codes": (c_int32, [_P, _P, _P, _P, c_int64, c_int64, c_int64, _P, c_int64, c_int64, _P, c_int64, _P]),
    "gdn_gemm_f32": (c_int32, [_P, _P, c_int64, c_int64, c_int64, _P, c_int64, c_int64, _P, c_int64, _P]),
    "gdn_conv": (c_int32, [_P, _P, c_int64, c_int64, _P, _P, c_int64, _P, _P, _P, _P]),
    "gdn_conv_state_update": (c_int32, [_P, _P, c_int64, c_int64, _P, _P]),
    "gdn_delta_rule": (c_int32, [_P, _P, _P, _P, c_int64, _P, _P, _P, _P, c_size_t, _P]),
    "gdn_delta_rule_scratch_size": (c_size_t, [_P, c_int64]),
    "gdn_delta_rule_noalloc": (c_int32, [_P, _P, _P, _P, c_int64, _P, _P, _P, _P]),
    "gdn_test_delta_wait_timeout": (c_int32, [_P, _P, _P, _P, c_int64, _P, c_size_t, ctypes.c_uint64, _P]),
    "gdn_gated_norm": (c_int32, [_P, _P, _P, c_int64, c_int64, _P, _P, _P, _P]),
}


class GdnError(RuntimeError):
    def __init__(self, name, code, msg):
        super().__init__(f"{name} returned {code}: {msg}")
        self.code = code


def header_functions() -> list:
    """Names of the functions ``include/gdn.h`` declares."""
    path = os.path.join(_build.INCLUDE, "gdn.h")
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(", text, flags=re.M)
    return [n for n in names if n not in ("if", "defined")]


class Lib:
    """The loaded library; each method has the C function's name and arguments."""

    def __init__(self, path: str):
        self.path = path
        self.dll = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(self.dll, name)
            fn.restype = res
            fn.argtypes = args

    def last_error(self) -> str:
        return self.dll.gdn_last_error().decode()

    def _call(self, name, *args, check=True):
        r = getattr(self.dll, name)(*args)
        if check and r != GDN_OK:
            raise GdnError(name, r, self.last_error())
        return r

    def __getattr__(self, name):
        if name in _SIGNATURES:
            status = _SIGNATURES[name][0] is c_int32     # size queries return sizes, not statuses
            return lambda *a, check=status: self._call(name, *a, check=check)
        raise AttributeError(name)


_LIBS = {}


def load(build: bool = False, debug: bool = False) -> Lib:
    """Load ``_lib/libgdn.so`` (building it first if ``build``), or with
    ``debug`` its debug variant ``_lib/libgdn_debug.so``: the same kernels with
    every global store's index checked (a failed check is skipped and reported
    by gdn_sync_status as GDN_EINDEX).  The two are separate libraries with
    separate device state; both may be loaded at once."""
    if debug not in _LIBS:
        if build:
            _build.build()
        path = _build.DEBUG_LIB if debug else _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libgdn is not built ({path} missing): run hybrid_gated_deltanet_q4k_gb300/build.py")
        _LIBS[debug] = Lib(path)
    return _LIBS[debug]


def ptr(t) -> int:
    """Device (or host) address of a torch tensor / numpy array, 0 for None."""
    if t is None:
        return 0
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    return t.ctypes.data


def stream_handle(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def make_layer_struct(spec, dev: dict, eps_l2=1e-6, eps_rms=1e-6, q_scale=None, gate_log_a=None, gate_b=None) -> GdnLayer:
    """Fill ``struct gdn_layer`` from a spec and device tensors w_in, w_out, conv_w, A_log, dt_bias, norm_w."""
    L = GdnLayer()
    L.hidden, L.n_qk_heads, L.n_v_heads = spec.hidden, spec.n_qk_heads, spec.n_v_heads
    L.dk, L.dv, L.conv_taps = spec.dk, spec.dv, 4
    L.wtype = GDN_W_Q4K if spec.wtype == "q4k" else GDN_W_F32
    L.w_in, L.w_out, L.conv_w = ptr(dev["w_in"]), ptr(dev["w_out"]), ptr(dev["conv_w"])
    L.A_log, L.dt_bias, L.norm_w = ptr(dev["A_log"]), ptr(dev["dt_bias"]), ptr(dev["norm_w"])
    L.gate_log_a, L.gate_b = ptr(gate_log_a), ptr(gate_b)
    L.eps_l2, L.eps_rms = eps_l2, eps_rms
    L.q_scale = spec.dk ** -0.5 if q_scale is None else q_scale
    return L
