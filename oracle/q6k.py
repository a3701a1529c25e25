"""GGUF Q6_K superblocks: decode to fp32 and a plain absmax encoder (oracle).

TEST INFRASTRUCTURE (see the package header).

The pages name Q6_K beside Q4_K as the second weight format the fused
dequant handles (sparkinfer PR #464 "fused Q4K/Q6K->int8 dequant +
token-parallel GDN conv ...", Summary, "Fused Q4_K/Q6_K -> int8-row
dequant": Q4_K_M files carry some tensors in Q6_K).  The block is the public
GGUF Q6_K block, 210 bytes for 256 weights:

    bytes   0-127  ql      low 4 bits of the 6-bit codes
    bytes 128-191  qh      high 2 bits of the 6-bit codes
    bytes 192-207  scales  sixteen int8 sub-block scales, one per 16 weights
    bytes 208-209  d       fp16 super-scale

Weight v (0..255) lies in half h = v // 128; with r = v % 128, group
g = r // 32 and lane l = r % 32 its low 4 bits are nibble g // 2 (0 = low,
1 = high) of ql[64h + 32(g % 2) + l] and its high 2 bits are bits 2g, 2g+1
of qh[32h + l].  The 6-bit code c = low | high << 4 stands for q = c - 32 in
-32..31, and the weight is  w = d * scales[v // 16] * q.

Decode rounding: |d| has at most 11 significant bits, |scale| <= 128 and
|q| <= 32, so d*scale*q is an integer multiple of d's last bit below 2^23 of
them: exact in fp32 in any order.  The oracle evaluates it in fp64 and casts.

The encoder is a plain reading (the pages give none, they only decode): per
sub-block of 16 weights step_j = max|x| / 31; d = max_j step_j / 127 rounded
to fp16 (a zero stored as +0); scale_j = clamp(rne(step_j / d), 0, 127);
q = clamp(rne(x / (d * scale_j)), -32, 31), a zero divisor giving 0; all in
IEEE fp32 with nearest-even rounding.
"""
from __future__ import annotations

import numpy as np

QK_K = 256
BLOCK_BYTES = 210


def _codes(ql: np.ndarray, qh: np.ndarray) -> np.ndarray:
    """6-bit codes (0..63) [..., 256] in weight order from ql [..., 128], qh [..., 64]."""
    lead = ql.shape[:-1]
    ql = ql.astype(np.int64).reshape(lead + (2, 2, 32))     # [.., half, g % 2, l]
    qh = qh.astype(np.int64).reshape(lead + (2, 32))        # [.., half, l]
    c = np.empty(lead + (2, 4, 32), np.int64)               # [.., half, g, l]
    for g in range(4):
        low = (ql[..., :, g % 2, :] >> (4 * (g // 2))) & 15
        high = (qh >> (2 * g)) & 3
        c[..., :, g, :] = low | (high << 4)
    return c.reshape(lead + (256,))


def unpack_q6k(blocks: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Decode Q6_K blocks (uint8 [rows, cols/256*210]) to float32 [rows, cols]."""
    assert cols % QK_K == 0
    nsb = cols // QK_K
    b = np.asarray(blocks, np.uint8).reshape(rows, nsb, BLOCK_BYTES)
    q = (_codes(b[..., 0:128], b[..., 128:192]) - 32).astype(np.float64)
    sc = b[..., 192:208].copy().view(np.int8).astype(np.float64)          # [rows, nsb, 16]
    d = b[..., 208:210].copy().view(np.float16)[..., 0].astype(np.float64)
    w = d[..., None, None] * sc[..., None] * q.reshape(rows, nsb, 16, 16)
    return w.reshape(rows, cols).astype(np.float32)


def _rne_f32(x: np.ndarray) -> np.ndarray:
    return np.rint(x.astype(np.float32)).astype(np.float32)


def pack_q6k(w: np.ndarray) -> np.ndarray:
    """Encode float32 [rows, cols] into Q6_K blocks uint8 [rows, cols/256*210]."""
    w = np.ascontiguousarray(w, np.float32)
    rows, cols = w.shape
    assert cols % QK_K == 0
    nsb = cols // QK_K
    f32 = np.float32
    x = w.reshape(rows, nsb, 16, 16)
    step = (np.abs(x).max(axis=-1) / f32(31)).astype(f32)              # [rows, nsb, 16]
    d16 = (step.max(axis=-1) / f32(127)).astype(f32).astype(np.float16)
    d16 = np.where(d16 == 0, np.float16(0), d16)
    d = d16.astype(f32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        sc = np.where(d > 0, np.clip(_rne_f32(step / np.where(d > 0, d, f32(1))), 0, 127), 0).astype(np.int64)
        ds = (d * sc.astype(f32)).astype(f32)[..., None]                 # exact products
        q = np.where(ds > 0, np.clip(_rne_f32(x / np.where(ds > 0, ds, f32(1))), -32, 31), 0).astype(np.int64)
    c = (q + 32).reshape(rows, nsb, 2, 4, 32)                           # [.., half, g, l]
    out = np.zeros((rows, nsb, BLOCK_BYTES), np.uint8)
    ql = np.zeros((rows, nsb, 2, 2, 32), np.int64)
    qh = np.zeros((rows, nsb, 2, 32), np.int64)
    for g in range(4):
        ql[..., :, g % 2, :] |= (c[..., :, g, :] & 15) << (4 * (g // 2))
        qh |= (c[..., :, g, :] >> 4) << (2 * g)
    out[..., 0:128] = ql.reshape(rows, nsb, 128).astype(np.uint8)
    out[..., 128:192] = qh.reshape(rows, nsb, 64).astype(np.uint8)
    out[..., 192:208] = sc.astype(np.int8).view(np.uint8)
    out[..., 208:210] = d16[..., None].view(np.uint8).reshape(rows, nsb, 2)
    return out.reshape(rows, nsb * BLOCK_BYTES)


def block_fields(blocks: np.ndarray, rows: int, cols: int) -> dict:
    """Decoded fields per superblock (for tests): d, scales [16], q [256] in -32..31."""
    nsb = cols // QK_K
    b = np.asarray(blocks, np.uint8).reshape(rows, nsb, BLOCK_BYTES)
    return {
        "d": b[..., 208:210].copy().view(np.float16)[..., 0],
        "scales": b[..., 192:208].copy().view(np.int8).astype(np.int64),
        "q": _codes(b[..., 0:128], b[..., 128:192]) - 32,
    }
