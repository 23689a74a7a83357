"""Pins of the oracle's storage formats and cold codec (CPU only).

Each check compares the oracle with something fixed outside it: hand-worked
bytes from the definitions on the pages (tests/golden), IEEE binary16
encodings, error bounds that follow from the quantiser's definition, and the
cosine fidelity the tiered-cache page reports for int4 cold blocks.
"""
import numpy as np
import pytest

from oracle import formats
from tests import golden



def test_f16_conversion_matches_ieee_encodings():
    for v, bits in golden.f16_values():
        got = formats.to_f16(np.float32(v)).view(np.uint16)
        assert int(got) == bits, (v, hex(int(got)), hex(bits))


@pytest.mark.parametrize("case", range(len(golden.q8_0_blocks())))
def test_q8_0_hand_worked_blocks(case):
    x, want = golden.q8_0_blocks()[case]
    got = formats.encode_rows("q8_0", np.array([x], dtype=np.float32), 1, 32)
    # one 34-byte block, padded to 36 (whole f32 words)
    assert got.shape == (1, 36)
    assert list(got[0, :34]) == want
    assert list(got[0, 34:]) == [0, 0]


def test_q8_0_divisor_blocks_tell_the_two_readings_apart():
    # The fixture's last four blocks code differently when the division uses
    # the stored f16 scale instead of the float32 amax/127: recomputing their
    # codes that other way must disagree with the expected bytes, so the
    # hand-worked pins above do decide which divisor the oracle uses.
    blocks = golden.q8_0_blocks()
    assert len(blocks) >= 8
    for x, want in blocks[4:]:
        x = np.array(x, dtype=np.float32)
        d16 = np.array(want[:2], dtype=np.uint8).view("<f2")[0]
        assert d16 != 0
        other = np.clip(np.rint(x / np.float32(d16)), -127, 127).astype(np.int8)
        assert list(other.view(np.uint8)) != want[2:]
        # and the stored scale is the f16 rounding of the float32 amax/127
        d32 = np.float32(np.abs(x).max()) / np.float32(127)
        assert np.float16(d32) == d16 and np.float32(d16) != d32


def test_q8_0_row_width_whole_blocks_in_whole_words():
    # "a whole number of Q8_0 blocks rounded up to whole f32 words"
    assert formats.row_bytes("q8_0", 1, 32) == 36
    assert formats.row_bytes("q8_0", 2, 64) == 136
    assert formats.row_bytes("q8_0", 8, 128) == 1088
    assert formats.row_bytes("q8_0", 3, 64) == 204
    assert formats.row_bytes("q8_0", 1, 96) == 104
    assert formats.row_bytes("f32", 3, 64) == 768
    assert formats.row_bytes("f16", 8, 128) == 2048
    with pytest.raises(ValueError):
        formats.row_bytes("q4_0", 8, 128)


def test_q8_0_heads_own_consecutive_blocks():
    # head h of a row owns blocks [h*d/32, (h+1)*d/32): a row whose head 1 is
    # a scaled copy of head 0 has block 2..3 equal to block 0..1 with scale x2
    rng = np.random.default_rng(0)
    h0 = rng.standard_normal(64).astype(np.float32)
    row = np.concatenate([h0, 2 * h0])[None]
    b = formats.encode_rows("q8_0", row, 2, 64)[0]
    blocks = b[:136].reshape(4, 34)
    assert (blocks[2, 2:] == blocks[0, 2:]).all() and (blocks[3, 2:] == blocks[1, 2:]).all()
    d0 = blocks[0, :2].view("<f2")[0]
    d2 = blocks[2, :2].view("<f2")[0]
    assert float(d2) == 2 * float(d0)


def test_q8_0_amax_maps_to_127_and_error_bound():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((500, 8 * 128)).astype(np.float32)
    enc = formats.encode_rows("q8_0", x, 8, 128)
    dec = formats.decode_rows("q8_0", enc, 8, 128)
    g = x.reshape(500, -1, 32).astype(np.float64)
    amax = np.abs(g).max(-1)
    d32 = amax / 127.0
    blocks = enc[:, :1088].reshape(500, 32, 34)
    q = blocks[:, :, 2:].view(np.int8).astype(np.int64)
    # the element of largest magnitude gets code +-127
    idx = np.abs(g).argmax(-1)
    top = np.take_along_axis(q, idx[..., None], -1)[..., 0]
    assert (np.abs(top) == 127).all()
    # |x - q*d16| <= d32/2 + 127*|d16 - d32| (code rounding plus f16 scale rounding)
    d16 = blocks[:, :, :2].copy().view("<f2")[..., 0].astype(np.float64)
    bound = d32 / 2 + 127 * np.abs(d16 - d32) + 1e-12
    err = np.abs(dec.reshape(500, -1, 32) - g).max(-1)
    assert (err <= bound).all()


def test_q8_0_exact_multiples_round_trip():
    d = 0.25
    k = np.arange(-127, 128, 8)
    x = np.zeros(32, dtype=np.float32)
    x[: len(k)] = k * d
    x[31] = 127 * d
    dec = formats.decode_rows("q8_0", formats.encode_rows("q8_0", x[None], 1, 32), 1, 32)[0]
    assert np.array_equal(dec, x.astype(np.float64))


@pytest.mark.parametrize("fmt", ["f32", "f16"])
def test_plain_formats_round_trip(fmt):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((7, 3 * 64)).astype(np.float32)
    dec = formats.decode_rows(fmt, formats.encode_rows(fmt, x, 3, 64), 3, 64)
    want = x if fmt == "f32" else x.astype(np.float16)
    assert np.array_equal(dec, want.astype(np.float64))


@pytest.mark.parametrize("case", range(4))
def test_int4_hand_worked_blocks(case):
    x, scale_b, nib_b, back = golden.int4_blocks()[case]
    scale, nib = formats.int4_quantize_block(np.array(x, dtype=np.float32))
    assert list(np.float32(scale).reshape(1).view(np.uint8)) == scale_b
    assert list(nib) == nib_b
    dq = formats.int4_dequantize_block(scale, nib, len(x), "f16")
    assert dq.astype(np.float64).tolist() == back


def test_int4_cosine_matches_reported_fidelity():
    # the tiered-cache page reports cosine ~0.99 against the unquantised block;
    # blocks of 16 slots x 4 heads x 256 dims of N(0,1) f16 values
    rng = np.random.default_rng(3)
    cos = []
    for _ in range(16):
        x = rng.standard_normal(16 * 4 * 256).astype(np.float32).astype(np.float16)
        s, nib = formats.int4_quantize_block(x)
        y = formats.int4_dequantize_block(s, nib, x.size, "f16").astype(np.float64)
        xx = x.astype(np.float64)
        cos.append(xx @ y / np.sqrt((xx @ xx) * (y @ y)))
    assert 0.98 <= min(cos) and max(cos) <= 0.995


def test_int4_error_bound_and_range():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal(4096) * 3).astype(np.float32)
    s, nib = formats.int4_quantize_block(x)
    codes = np.empty(2 * nib.size, dtype=np.int64)
    codes[0::2] = nib & 15
    codes[1::2] = nib >> 4
    assert codes.min() >= 1 and codes.max() <= 15  # |x| <= amax keeps q in [-7, 7]
    y = formats.int4_dequantize_block(s, nib, x.size, "f32").astype(np.float64)
    assert np.abs(y - x).max() <= float(s) / 2 * (1 + 1e-6)
    assert float(s) == float(np.float32(np.abs(x).max()) / np.float32(7))
