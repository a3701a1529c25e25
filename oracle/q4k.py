"""GGUF Q4_K superblocks: decode to fp32 and a plain min-max encoder (oracle).

TEST INFRASTRUCTURE (see the package header).

The pages name the format only as "superblocks" (sparkinfer PR #464 "fused
Q4K/Q6K->int8 dequant + token-parallel GDN conv ...", Summary, "Fused
Q4_K/Q6_K -> int8-row dequant": the kernel "decodes superblocks in registers").
The block is the public GGUF Q4_K block, 144 bytes for 256 weights:

    bytes 0-1    d      fp16, super-scale of the sub-block scales
    bytes 2-3    dmin   fp16, super-scale of the sub-block mins
    bytes 4-15   12 bytes holding eight 6-bit scales sc_j and eight 6-bit mins m_j
    bytes 16-143 128 bytes of 4-bit codes

Sub-block j (32 weights) decodes as  w = d*sc_j*q - dmin*m_j,  q in 0..15.
6-bit fields: for j < 4, sc_j = s[j] & 63 and m_j = s[j+4] & 63; for j >= 4,
sc_j = (s[j+4] & 15) | ((s[j-4] >> 6) << 4) and m_j = (s[j+4] >> 4) | ((s[j] >> 6) << 4).
Codes: weight 64p + l (l < 32) is the low nibble of qs[32p + l] (sub-block 2p);
weight 64p + 32 + l is its high nibble (sub-block 2p + 1).

Decode rounding: the decoded value is the exact real d*sc*q - dmin*m rounded
once to fp32 (nearest-even).  d*sc*q and dmin*m are exact in fp64, and their
difference is exact in fp64 too: fp16 values lie between 2^-24 and 2^16 and
sc*q < 2^10, so every bit of either term falls within a 50-bit window.  fp64
evaluation followed by one cast to fp32 is therefore that single rounding.

The encoder is a plain reading (the pages give none): per sub-block the
min-max range [min(0, min x), max x] is split into 15 steps; d and dmin are the
largest sub-block scale and min divided by 63, rounded to fp16 (a zero of
either sign stored as +0); sc_j, m_j and the codes are nearest-even roundings
clamped to their ranges, all in fp32.
"""
from __future__ import annotations

import numpy as np

QK_K = 256
BLOCK_BYTES = 144


def _scale_min_6bit(sb: np.ndarray):
    """Unpack the 12 scale bytes [..., 12] into sc, m [..., 8] (int64)."""
    s = sb.astype(np.int64)
    sc = np.empty(s.shape[:-1] + (8,), np.int64)
    m = np.empty_like(sc)
    for j in range(4):
        sc[..., j] = s[..., j] & 63
        m[..., j] = s[..., j + 4] & 63
    for j in range(4, 8):
        sc[..., j] = (s[..., j + 4] & 15) | ((s[..., j - 4] >> 6) << 4)
        m[..., j] = (s[..., j + 4] >> 4) | ((s[..., j] >> 6) << 4)
    return sc, m


def _codes(qs: np.ndarray) -> np.ndarray:
    """4-bit codes [..., 128 bytes] -> [..., 256] in weight order."""
    q = qs.astype(np.int64).reshape(qs.shape[:-1] + (4, 32))
    lo = q & 15
    hi = q >> 4
    return np.concatenate([lo[..., None, :], hi[..., None, :]], axis=-2).reshape(qs.shape[:-1] + (256,))


def unpack_q4k(blocks: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Decode Q4_K blocks (uint8 [rows, cols/256*144]) to float32 [rows, cols]."""
    assert cols % QK_K == 0
    nsb = cols // QK_K
    b = np.asarray(blocks, np.uint8).reshape(rows, nsb, BLOCK_BYTES)
    d = b[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    dmin = b[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    sc, m = _scale_min_6bit(b[..., 4:16])
    q = _codes(b[..., 16:144]).reshape(rows, nsb, 8, 32).astype(np.float64)
    w = (d[..., None, None] * sc[..., None].astype(np.float64)) * q - (dmin[..., None, None] * m[..., None].astype(np.float64))
    return w.reshape(rows, cols).astype(np.float32)


def _rne_f32(x: np.ndarray) -> np.ndarray:
    return np.rint(x.astype(np.float32)).astype(np.float32)


def pack_q4k(w: np.ndarray) -> np.ndarray:
    """Encode float32 [rows, cols] into Q4_K blocks uint8 [rows, cols/256*144]."""
    w = np.ascontiguousarray(w, np.float32)
    rows, cols = w.shape
    assert cols % QK_K == 0
    nsb = cols // QK_K
    x = w.reshape(rows, nsb, 8, 32)
    f32 = np.float32
    mn = np.minimum(x.min(axis=-1), f32(0))                 # [rows, nsb, 8]
    mx = x.max(axis=-1)
    scale = ((mx - mn).astype(f32) / f32(15)).astype(f32)   # step of each sub-block
    mins = (-mn).astype(f32)
    d16 = (scale.max(axis=-1) / f32(63)).astype(f32).astype(np.float16)
    dm16 = (mins.max(axis=-1) / f32(63)).astype(f32).astype(np.float16)
    d16 = np.where(d16 == 0, np.float16(0), d16)     # a zero super-scale of either sign is stored as +0
    dm16 = np.where(dm16 == 0, np.float16(0), dm16)
    d = d16.astype(f32)[..., None]
    dm = dm16.astype(f32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        sc = np.where(d > 0, np.clip(_rne_f32(scale / np.where(d > 0, d, f32(1))), 0, 63), 0).astype(np.int64)
        mm = np.where(dm > 0, np.clip(_rne_f32(mins / np.where(dm > 0, dm, f32(1))), 0, 63), 0).astype(np.int64)
        ds = (d * sc.astype(f32)).astype(f32)[..., None]      # exact products
        dms = (dm * mm.astype(f32)).astype(f32)[..., None]
        num = (x + dms).astype(f32)
        q = np.where(ds > 0, np.clip(_rne_f32(num / np.where(ds > 0, ds, f32(1))), 0, 15), 0).astype(np.int64)
    out = np.zeros((rows, nsb, BLOCK_BYTES), np.uint8)
    out[..., 0:2] = d16[..., None].view(np.uint8).reshape(rows, nsb, 2)
    out[..., 2:4] = dm16[..., None].view(np.uint8).reshape(rows, nsb, 2)
    s = np.zeros((rows, nsb, 12), np.int64)
    for j in range(4):
        s[..., j] = (sc[..., j] & 63) | ((sc[..., j + 4] >> 4) << 6)
        s[..., j + 4] = (mm[..., j] & 63) | ((mm[..., j + 4] >> 4) << 6)
        s[..., j + 8] = (sc[..., j + 4] & 15) | ((mm[..., j + 4] & 15) << 4)
    out[..., 4:16] = s.astype(np.uint8)
    qv = q.reshape(rows, nsb, 4, 2, 32)                      # [.., group p, lo/hi, l]
    out[..., 16:144] = (qv[..., 0, :] | (qv[..., 1, :] << 4)).reshape(rows, nsb, 128).astype(np.uint8)
    return out.reshape(rows, nsb * BLOCK_BYTES)


def block_fields(blocks: np.ndarray, rows: int, cols: int) -> dict:
    """Decoded header fields per superblock (for tests): d, dmin, sc, m, q."""
    nsb = cols // QK_K
    b = np.asarray(blocks, np.uint8).reshape(rows, nsb, BLOCK_BYTES)
    sc, m = _scale_min_6bit(b[..., 4:16])
    return {
        "d": b[..., 0:2].copy().view(np.float16)[..., 0],
        "dmin": b[..., 2:4].copy().view(np.float16)[..., 0],
        "sc": sc,
        "m": m,
        "q": _codes(b[..., 16:144]).reshape(rows, nsb, 8, 32),
    }
