"""Pins for the oracle's Q6_K decode and encoder (closed forms, hand-decoded
bit positions, brute force, bounds, planted mistakes)."""
import numpy as np
import pytest

from oracle import q6k

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _block(d, scales16, ql128, qh64):
    b = np.zeros(210, np.uint8)
    b[0:128] = np.asarray(ql128, np.uint8)
    b[128:192] = np.asarray(qh64, np.uint8)
    b[192:208] = np.asarray(scales16, np.int8).view(np.uint8)
    b[208:210] = np.array([d], np.float16).view(np.uint8)
    return b[None, :]


# ----------------------------------------------------------------- decode pins

def check_decode_closed_forms(unpack):
    # every 6-bit code 63 (q = 31), every scale 127: every weight is 31*127*d
    w = unpack(_block(2.0 ** -12, [127] * 16, [0xFF] * 128, [0xFF] * 64), 1, 256)
    assert np.all(w == np.float32(31 * 127 * 2.0 ** -12))
    # every code 0 (q = -32), scales -128: every weight is (-32)(-128) d = 4096 d
    w = unpack(_block(0.5, [-128] * 16, [0] * 128, [0] * 64), 1, 256)
    assert np.all(w == np.float32(4096 * 0.5))
    # code 32 (q = 0): low nibble 0, high bits 2 -> zero for any scale
    w = unpack(_block(3.0, [77] * 16, [0] * 128, [0xAA] * 64), 1, 256)
    assert np.all(w == 0)


def check_decode_bit_positions(unpack):
    # Background code 32 (q = 0: ql nibbles 0, qh pairs 2 = 0b10).  Raising the
    # low nibble of one ql byte to 1, or one qh bit pair from 2 to 3, makes
    # exactly one weight nonzero (q = 1 or q = 16), at the position the layout
    # gives; the scale of weight v is scales[v // 16] = v // 16 + 1.
    scales = np.arange(1, 17)
    for byte in [0, 7, 31, 32, 63, 64, 100, 127]:
        h, g1, l = byte // 64, (byte % 64) // 32, byte % 32
        for nib in (0, 1):
            ql = np.zeros(128, np.uint8)
            ql[byte] = 1 << (4 * nib)
            w = unpack(_block(1.0, scales, ql, [0xAA] * 64), 1, 256)[0]
            v = 128 * h + 32 * (g1 + 2 * nib) + l
            assert list(np.flatnonzero(w)) == [v]
            assert w[v] == np.float32(1 * (v // 16 + 1))
    for byte in [0, 5, 31, 32, 50, 63]:
        h, l = byte // 32, byte % 32
        for g in range(4):
            qh = np.full(64, 0xAA, np.uint8)
            qh[byte] |= 1 << (2 * g)                  # pair g: 2 -> 3
            w = unpack(_block(1.0, scales, np.zeros(128, np.uint8), qh), 1, 256)[0]
            v = 128 * h + 32 * g + l
            assert list(np.flatnonzero(w)) == [v]
            assert w[v] == np.float32(16 * (v // 16 + 1))


def check_decode_exact_products(unpack):
    # d with all 11 significant bits set, scale -127, q = -31 (code 1): the
    # exact product 0x7FF * 2^-10 * 127 * 31 fits fp32 exactly
    d = float(np.float16(2 - 2 ** -10))
    ql = np.zeros(128, np.uint8)
    ql[:] = 0x11                                      # low nibbles 1 everywhere
    w = unpack(_block(d, [-127] * 16, ql, [0] * 64), 1, 256)[0]
    assert np.all(w == np.float32(d * -127 * -31))
    assert float(w[0]) == d * 127 * 31                # no rounding happened


@pytest.mark.parametrize("check", [check_decode_closed_forms, check_decode_bit_positions,
                                   check_decode_exact_products])
def test_decode_pins(check):
    check(q6k.unpack_q6k)


def test_planted_high_bit_shift_is_caught(monkeypatch):
    """A decode that takes the high bits of group g from bits g, g+1 of qh
    (instead of 2g, 2g+1) must fail the bit-position pin."""
    def wrong(ql, qh):
        lead = ql.shape[:-1]
        qlr = ql.astype(np.int64).reshape(lead + (2, 2, 32))
        qhr = qh.astype(np.int64).reshape(lead + (2, 32))
        c = np.empty(lead + (2, 4, 32), np.int64)
        for g in range(4):
            c[..., :, g, :] = ((qlr[..., :, g % 2, :] >> (4 * (g // 2))) & 15) | (((qhr >> g) & 3) << 4)
        return c.reshape(lead + (256,))
    monkeypatch.setattr(q6k, "_codes", wrong)
    with pytest.raises(AssertionError):
        check_decode_bit_positions(q6k.unpack_q6k)


def test_planted_missing_offset_is_caught():
    """A decode without the -32 offset must fail the closed forms."""
    def no_offset(blocks, rows, cols):
        b = np.asarray(blocks, np.uint8).reshape(rows, -1, 210)
        c = q6k._codes(b[..., :128], b[..., 128:192]).astype(np.float64)
        sc = b[..., 192:208].copy().view(np.int8).astype(np.float64)
        d = b[..., 208:210].copy().view(np.float16)[..., 0].astype(np.float64)
        return (d[..., None, None] * sc[..., None] * c.reshape(rows, -1, 16, 16)).reshape(rows, cols).astype(np.float32)
    with pytest.raises(AssertionError):
        check_decode_closed_forms(no_offset)


def test_planted_scale_per_32_is_caught():
    """A decode that applies one scale per 32 weights must fail the bit-position pin."""
    def per32(blocks, rows, cols):
        b = np.asarray(blocks, np.uint8).reshape(rows, -1, 210)
        q = (q6k._codes(b[..., :128], b[..., 128:192]) - 32).astype(np.float64)
        sc = b[..., 192:208].copy().view(np.int8).astype(np.float64)
        d = b[..., 208:210].copy().view(np.float16)[..., 0].astype(np.float64)
        s256 = np.repeat(sc[..., :8], 32, axis=-1)
        return (d[..., None] * s256 * q).reshape(rows, cols).astype(np.float32)
    with pytest.raises(AssertionError):
        check_decode_bit_positions(per32)


# ----------------------------------------------------------------- encoder pins

def _grid_blocks(rng, rows, nsb):
    """Blocks on the encoder's own grid: per sub-block the code magnitudes
    reach 31 (so its step is the decoded scale) and one scale per superblock
    is 127 (so d is recovered)."""
    out = np.zeros((rows, nsb, 210), np.uint8)
    for r in range(rows):
        for s in range(nsb):
            sc = rng.integers(1, 128, size=16)
            sc[rng.integers(16)] = 127
            q = rng.integers(-31, 32, size=(16, 16))
            q[:, 0] = np.where(rng.random(16) < 0.5, 31, -31)
            d = float(np.float16(rng.uniform(1e-5, 1e-3)))
            c = (q + 32).reshape(2, 4, 32)
            ql = np.zeros((2, 2, 32), np.int64)
            qh = np.zeros((2, 32), np.int64)
            for g in range(4):
                ql[:, g % 2, :] |= (c[:, g, :] & 15) << (4 * (g // 2))
                qh |= (c[:, g, :] >> 4) << (2 * g)
            out[r, s] = _block(d, sc, ql.reshape(128), qh.reshape(64))[0]
    return out.reshape(rows, nsb * 210)


def test_pack_recovers_grid_blocks_exactly():
    rng = np.random.default_rng(5)
    blocks = _grid_blocks(rng, 3, 4)
    w = q6k.unpack_q6k(blocks, 3, 1024)
    assert np.array_equal(q6k.pack_q6k(w), blocks)


def test_pack_codes_and_scales_are_nearest_brute_force():
    rng = np.random.default_rng(9)
    w = rng.normal(0, 0.02, size=(4, 512)).astype(np.float32)
    f = q6k.block_fields(q6k.pack_q6k(w), 4, 512)
    d = f["d"].astype(np.float32)
    x = w.reshape(4, 2, 16, 16)
    for r in range(4):
        for s in range(2):
            step = np.abs(x[r, s]).max(-1) / np.float32(31)
            for j in range(16):
                ds = np.float32(d[r, s] * f["scales"][r, s, j])
                cand = np.arange(-32, 32, dtype=np.float64) * float(ds)
                for i in range(16):
                    err = np.abs(cand - float(x[r, s, j, i]))
                    assert err[f["q"][r, s, 16 * j + i] + 32] <= err.min() + 1e-6 * float(ds) + 1e-12
                t = float(step[j]) / float(d[r, s])
                cs = np.abs(np.arange(128) - t)
                assert cs[f["scales"][r, s, j]] <= cs.min() + 1e-5


def test_pack_reconstruction_error_bound():
    rng = np.random.default_rng(13)
    w = rng.normal(0, 0.02, size=(8, 1024)).astype(np.float32)
    blocks = q6k.pack_q6k(w)
    deq = q6k.unpack_q6k(blocks, 8, 1024).astype(np.float64)
    f = q6k.block_fields(blocks, 8, 1024)
    x = w.astype(np.float64).reshape(8, 4, 16, 16)
    ds = f["d"].astype(np.float64)[..., None] * f["scales"]
    step = np.abs(x).max(-1) / 31
    # inside the representable range the error is half a step; the rounding of
    # the scale index moves the range's end by at most 31 |step - ds|
    bound = ds / 2 + 31 * np.abs(step - ds) + 1e-9
    assert np.all(np.abs(x - deq.reshape(x.shape)) <= bound[..., None])
    assert np.linalg.norm(x.ravel() - deq.ravel()) / np.linalg.norm(x) < 0.03   # 6-bit codes


def test_pack_zero_and_constant_rows():
    w = np.zeros((2, 256), np.float32)
    w[1] = -0.25
    deq = q6k.unpack_q6k(q6k.pack_q6k(w), 2, 256)
    assert np.all(deq[0] == 0)
    assert np.allclose(deq[1], -0.25, rtol=2 ** -9)
