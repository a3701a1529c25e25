"""Pins for the oracle's Q4_K decode and encoder (closed forms, brute force, bounds)."""
import numpy as np
import pytest

from oracle import q4k

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _block(d, dmin, scales12, qs128):
    b = np.zeros(144, np.uint8)
    b[0:2] = np.array([d], np.float16).view(np.uint8)
    b[2:4] = np.array([dmin], np.float16).view(np.uint8)
    b[4:16] = np.asarray(scales12, np.uint8)
    b[16:144] = np.asarray(qs128, np.uint8)
    return b[None, :]


# ----------------------------------------------------------------- decode pins

def check_decode_closed_forms(unpack):
    # all codes 15, every sub-block scale 63, mins 0: every weight is 945*d.
    sc = [0xFF] * 4 + [0x00] * 4 + [0x0F] * 4     # sc_j = 63 for all j, m_j = 0
    blk = _block(2.0 ** -10, 0.5, sc, [0xFF] * 128)
    w = unpack(blk, 1, 256)
    assert np.all(w == np.float32(945 * 2.0 ** -10))
    # all codes 0, mins 63: every weight is -63*dmin.
    sc = [0x00] * 4 + [0xFF] * 4 + [0xF0] * 4     # sc_j = 0, m_j = 63 for all j
    blk = _block(1.0, 2.0 ** -6, sc, [0] * 128)
    w = unpack(blk, 1, 256)
    assert np.all(w == np.float32(-63 * 2.0 ** -6))


def check_decode_scale_bits(unpack):
    # Hand-decoded 6-bit fields of the GGUF Q4_K layout:
    #   s = C1 02 03 04 05 06 07 08 9A 00 00 00
    #   sc0 = 0xC1 & 63 = 1, m0 = 0x05 & 63 = 5
    #   sc4 = (0x9A & 15) | ((0xC1 >> 6) << 4) = 10 | 48 = 58
    #   m4  = (0x9A >> 4) | ((0x05 >> 6) << 4) = 9
    s = [0xC1, 0x02, 0x03, 0x04, 0x05, 0x06, 0x07, 0x08, 0x9A, 0x00, 0x00, 0x00]
    qs = np.zeros(128, np.uint8)
    qs[0] = 0x01          # weight 0 (sub-block 0) code 1, weight 32 (sub-block 1) code 0
    qs[64] = 0x01         # weight 128 (sub-block 4) code 1
    w = unpack(_block(1.0, 1.0, s, qs), 1, 256)
    assert w[0, 0] == np.float32(1 * 1 - 5)         # d*sc0*1 - dmin*m0
    assert w[0, 128] == np.float32(58 * 1 - 9)      # d*sc4*1 - dmin*m4
    assert w[0, 129] == np.float32(-9)              # code 0 in sub-block 4
    # sc1 = 2, m1 = 6: weight 32 has code 0 -> -6
    assert w[0, 32] == np.float32(-6)


def check_decode_nibble_positions(unpack):
    # One code of value 1 at byte b, low or high nibble; all scales 1, mins 0:
    # exactly one decoded weight is 1, at 64*(b//32) + (b%32) (+32 for the high nibble).
    s = [1 | 0] * 4 + [0] * 4 + [0x01] * 4        # sc_j = 1 for all j, m_j = 0
    for b in [0, 5, 31, 32, 77, 127]:
        for hi in (0, 1):
            qs = np.zeros(128, np.uint8)
            qs[b] = (1 << 4) if hi else 1
            w = unpack(_block(1.0, 0.0, s, qs), 1, 256)[0]
            nz = np.flatnonzero(w)
            assert list(nz) == [64 * (b // 32) + (b % 32) + 32 * hi]
            assert w[nz[0]] == 1.0


def check_decode_single_rounding(unpack):
    # d = 1 + 2^-10 (fp16), sc = 63, q = 15, dmin*m chosen so that the exact real
    # d*sc*q - dmin*m needs more than 24 bits: the result must be its single
    # nearest-even fp32 rounding.
    d = float(np.float16(1 + 2 ** -10))
    dmin = float(np.float16(2.0 ** -24))           # smallest fp16 subnormal
    s = [0xFF] * 4 + [0x01] * 4 + [0x0F] * 4      # sc_j = 63; m_j = 1 for j < 4, 0 for j >= 4
    w = unpack(_block(d, dmin, s, [0xFF] * 128), 1, 256)[0]
    exact = d * 63 * 15 - dmin * 1                   # 34 significant bits: exact in fp64
    assert w[0] == np.float32(exact)
    assert w[32] == w[0]                            # sub-block 1: sc = 63, m = 1 as well
    assert w[128] == np.float32(d * 945)            # sub-block 4: sc = 63, m = 0


@pytest.mark.parametrize("check", [check_decode_closed_forms, check_decode_scale_bits,
                                   check_decode_nibble_positions, check_decode_single_rounding])
def test_decode_pins(check):
    check(q4k.unpack_q4k)


def test_planted_nibble_swap_is_caught():
    """A decode that swaps low and high nibbles must fail the nibble pin."""
    def swapped(blocks, rows, cols):
        b = np.array(blocks, np.uint8, copy=True).reshape(rows, -1, 144)
        qs = b[..., 16:]
        b[..., 16:] = ((qs & 15) << 4) | (qs >> 4)
        return q4k.unpack_q4k(b.reshape(rows, -1), rows, cols)
    with pytest.raises(AssertionError):
        check_decode_nibble_positions(swapped)


def test_planted_scale_bit_mixup_is_caught(monkeypatch):
    """A decode that takes m_j's high bits from the scale byte must fail the field pin."""
    orig = q4k._scale_min_6bit

    def wrong(sb):
        sc, m = orig(sb)
        s = sb.astype(np.int64)
        for j in range(4, 8):
            m[..., j] = (s[..., j + 4] >> 4) | ((s[..., j - 4] >> 6) << 4)
        return sc, m
    monkeypatch.setattr(q4k, "_scale_min_6bit", wrong)
    with pytest.raises(AssertionError):
        check_decode_scale_bits(q4k.unpack_q4k)


# ----------------------------------------------------------------- encoder pins

def _grid_blocks(rng, rows, nsb):
    """Blocks whose sub-blocks each hold codes 0 and 15, with max sc = max m = 63."""
    out = np.zeros((rows, nsb, 144), np.uint8)
    for r in range(rows):
        for s in range(nsb):
            sc = rng.integers(1, 64, size=8)
            m = rng.integers(0, 64, size=8)
            sc[rng.integers(8)] = 63
            m[rng.integers(8)] = 63
            q = rng.integers(0, 16, size=(8, 32))
            q[:, 0] = 0
            q[:, 1] = 15
            d = float(np.float16(rng.uniform(1e-4, 1e-2)))
            dm = float(np.float16(rng.uniform(1e-4, 1e-2)))
            s12 = np.zeros(12, np.int64)
            for j in range(4):
                s12[j] = sc[j] | ((sc[j + 4] >> 4) << 6)
                s12[j + 4] = m[j] | ((m[j + 4] >> 4) << 6)
                s12[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
            qs = np.zeros(128, np.int64)
            for p in range(4):
                qs[32 * p:32 * p + 32] = q[2 * p] | (q[2 * p + 1] << 4)
            out[r, s] = _block(d, dm, s12, qs)[0]
    return out.reshape(rows, nsb * 144)


def test_pack_recovers_grid_blocks_exactly():
    rng = np.random.default_rng(7)
    blocks = _grid_blocks(rng, 3, 4)
    w = q4k.unpack_q4k(blocks, 3, 1024)
    assert np.array_equal(q4k.pack_q4k(w), blocks)


def test_pack_codes_are_nearest_brute_force():
    rng = np.random.default_rng(3)
    w = rng.normal(0, 0.02, size=(4, 512)).astype(np.float32)
    f = q4k.block_fields(q4k.pack_q4k(w), 4, 512)
    d = f["d"].astype(np.float32)
    dm = f["dmin"].astype(np.float32)
    x = w.reshape(4, 2, 8, 32)
    for r in range(4):
        for s in range(2):
            for j in range(8):
                ds = np.float32(d[r, s] * f["sc"][r, s, j])
                dms = np.float32(dm[r, s] * f["m"][r, s, j])
                cand = np.arange(16, dtype=np.float64) * float(ds) - float(dms)   # every code's value
                for i in range(32):
                    err = np.abs(cand - float(x[r, s, j, i]))
                    chosen = err[f["q"][r, s, j, i]]
                    assert chosen <= err.min() + 1e-6 * float(ds) + 1e-9
            # scale indices nearest to each sub-block's min-max step
            mn = np.minimum(x[r, s].min(-1), 0)
            step = (x[r, s].max(-1) - mn) / np.float32(15)
            for j in range(8):
                if d[r, s] > 0:
                    t = float(step[j]) / float(d[r, s])
                    cand = np.abs(np.arange(64) - t)
                    assert cand[f["sc"][r, s, j]] <= cand.min() + 1e-5


def test_pack_reconstruction_error_bound():
    rng = np.random.default_rng(11)
    w = rng.normal(0, 0.02, size=(8, 1024)).astype(np.float32)
    blocks = q4k.pack_q4k(w)
    deq = q4k.unpack_q4k(blocks, 8, 1024)
    f = q4k.block_fields(blocks, 8, 1024)
    x = w.reshape(8, 4, 8, 32).astype(np.float64)
    dq = deq.reshape(8, 4, 8, 32).astype(np.float64)
    ds = f["d"].astype(np.float64)[..., None] * f["sc"]
    dms = f["dmin"].astype(np.float64)[..., None] * f["m"]
    mn = np.minimum(x.min(-1), 0)
    step = (x.max(-1) - mn) / 15
    # the representable range [-dms, 15 ds - dms] differs from [mn, mx] by the
    # rounding of the scale and min indices; inside it the error is <= ds/2.
    slack = 15 * np.abs(step - ds) + np.abs(-mn - dms)
    bound = ds / 2 + slack + 1e-7
    assert np.all(np.abs(x - dq) <= bound[..., None])
    rel = np.linalg.norm(x - dq) / np.linalg.norm(x)
    assert rel < 0.12      # 4-bit codes: about step/sqrt(12) per weight


def test_pack_zero_and_constant_rows():
    w = np.zeros((2, 256), np.float32)
    w[1] = -0.5
    blocks = q4k.pack_q4k(w)
    deq = q4k.unpack_q4k(blocks, 2, 256)
    assert np.all(deq[0] == 0)
    assert np.allclose(deq[1], -0.5, rtol=2 ** -10)
