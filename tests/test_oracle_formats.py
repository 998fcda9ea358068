"""Pins of the oracle's number formats against hand-derived tables and
closed forms (no GPU)."""

import math
import os

import numpy as np
import pytest

from oracle import formats as F


def _rows(path):
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def _val(s):
    return float("nan") if s == "nan" else float(s)


def test_e4m3_table(golden_dir):
    rows = list(_rows(os.path.join(golden_dir, "e4m3_codes.txt")))
    assert len(rows) >= 20
    for r in rows:
        code, want = int(r[0], 16), _val(r[1])
        got = float(F.e4m3_decode(code))
        if math.isnan(want):
            assert math.isnan(got)
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (hex(code), got, want)


def test_e4m3_structure():
    """Properties of the whole code space that a wrong bias, mantissa width or
    subnormal rule would break."""
    pos = F.e4m3_decode(np.arange(0x7F))
    assert np.all(np.diff(pos) > 0)  # strictly increasing over 0x00..0x7E
    assert pos[-1] == 448.0 and pos[1] == 2.0 ** -9
    assert np.isnan(F.e4m3_decode(0x7F)) and np.isnan(F.e4m3_decode(0xFF))
    neg = F.e4m3_decode(np.arange(0x80, 0xFF))
    assert np.array_equal(neg, -pos)
    # every binade e>=1 holds 8 values spaced 2^(e-10)
    for e in range(1, 15):
        v = pos[8 * e: 8 * e + 8]
        assert np.allclose(np.diff(v), 2.0 ** (e - 10))
    assert len(np.unique(pos)) == 127


def test_e2m1_table(golden_dir):
    for r in _rows(os.path.join(golden_dir, "e2m1_codes.txt")):
        code, want = int(r[0], 16), float(r[1])
        got = float(F.e2m1_decode(code))
        assert got == want and math.copysign(1, got) == math.copysign(1, want)


def test_rn_conversions(golden_dir):
    for fmt, x, want, *_ in _rows(os.path.join(golden_dir, "rn_cases.txt")):
        xv = np.float32(float(x)).astype(np.float64)
        enc = F.e2m1_encode_rn if fmt == "e2m1" else F.e4m3_encode_rn
        got = int(enc(np.array([xv]))[0])
        assert got == int(want, 16), (fmt, x, hex(got), want)


def test_rn_is_nearest():
    """Brute force: the encoded value is a nearest representable value for a
    dense sweep of inputs (checks the nearest-search independently of ties)."""
    xs = np.linspace(-500, 500, 200001)
    for enc, dec, mags in ((F.e4m3_encode_rn, F.e4m3_decode, F.E4M3_MAG),
                           (F.e2m1_encode_rn, F.e2m1_decode, F.E2M1_MAG)):
        got = dec(enc(xs))
        best = np.min(np.abs(np.abs(xs)[:, None] - mags[None, :]), axis=1)
        sat = np.abs(xs) >= mags[-1]
        assert np.all(np.abs(np.abs(got) - np.abs(xs))[~sat] <= best[~sat] + 0.0)
        assert np.all(np.abs(got[sat]) == mags[-1])
        assert np.all(np.sign(got[got != 0]) == np.sign(xs[got != 0]))


def _blocks(golden_dir):
    for r in _rows(os.path.join(golden_dir, "nvfp4_blocks.txt")):
        name, bytes_, scale, ts = r[0], r[1], r[2], r[3]
        vals = [float(v) for v in r[4:]]
        packed = np.array([int(b, 16) for b in bytes_.split(",")], dtype=np.uint8)
        yield name, packed, int(scale, 16), float(ts), np.array(vals)


def test_nvfp4_hand_blocks(golden_dir):
    n = 0
    for name, packed, scale, ts, want in _blocks(golden_dir):
        got = F.nvfp4_dequant(packed[None, :], np.array([[scale]], dtype=np.uint8), np.float32(ts), 16)[0]
        assert np.array_equal(got, want), (name, got, want)
        assert np.array_equal(np.signbit(got), np.signbit(want)), name
        n += 1
    assert n == 6


def test_nibble_order():
    packed = np.array([[0x21, 0x43]], dtype=np.uint8)
    assert F.unpack_nibbles(packed, 4).tolist() == [[1, 2, 3, 4]]
    assert np.array_equal(F.pack_nibbles(F.unpack_nibbles(packed, 4)), packed)


def test_rb_closed_forms():
    # bf16 grid near 1: spacing 2^-7; near 256: spacing 2
    assert F.rb(1.0 + 2 ** -8) == 1.0  # tie -> even (1.0)
    assert F.rb(1.0 + 3 * 2 ** -8) == 1.0 + 2 ** -6  # tie -> even mantissa
    assert F.rb(1.0 + 2 ** -8 + 2 ** -30) == 1.0 + 2 ** -7  # above the tie
    assert F.rb(257.0) == 256.0 and F.rb(259.0) == 260.0
    assert F.rb(-3.0e38) == -2.9969737e38 or abs(F.rb(-3.0e38) + 3.0e38) / 3e38 < 2 ** -8
    assert F.rb(1e-40) != 0 and abs(F.rb(1e-40) - 1e-40) <= 2 ** -134
    assert F.rb(0.0) == 0.0 and np.isnan(F.rb(np.nan))
    # no double rounding: a value that rounds differently via fp32 first
    x = 1.0 + 2 ** -8 + 2 ** -40  # fp32 would round it to the tie 1+2^-8, then to 1.0
    assert F.rb(x) == 1.0 + 2 ** -7


def test_q4_cases():
    z = np.zeros(16)
    b = z.copy(); b[0] = 6.0
    codes, sc, vals = F.q4(b)
    assert sc.tolist() == [0x38] and codes[0] == 7 and np.all(codes[1:] == 0) and vals[0] == 6.0
    b = z.copy(); b[:3] = [3.0, -1.5, 0.75]
    codes, sc, vals = F.q4(b)
    assert sc.tolist() == [0x30] and codes[:3].tolist() == [7, 0xD, 3]
    assert vals[:3].tolist() == [3.0, -1.5, 0.75]
    # amax / 6 below half the smallest subnormal scale -> zero block
    b = z.copy(); b[5] = 0.001
    codes, sc, vals = F.q4(b)
    assert np.all(vals == 0)
    # amax 7 -> scale rounds down to 1.125; 7/1.125 saturates to 6 -> 6.75
    b = z.copy(); b[2] = 7.0
    codes, sc, vals = F.q4(b)
    assert sc.tolist() == [0x39] and vals[2] == 6.75
    # all-zero block
    codes, sc, vals = F.q4(z)
    assert sc.tolist() == [0] and np.all(codes == 0)
    # two independent blocks along the axis.  0.5/6 = 0.0833.. lies between
    # E4M3 0.078125 (0x1A) and 0.0859375 (0x1B), nearer the latter; then
    # 0.5/0.0859375 = 5.82 -> E2M1 6 -> 0.515625.  4/6 = 0.666.. -> 0.6875
    # (0x33, between 0.625 and 0.6875); 4/0.6875 = 5.82 -> 6 -> 4.125.
    x = np.concatenate([np.full(16, 0.5), np.full(16, 4.0)])
    codes, sc, vals = F.q4(x)
    assert sc.tolist() == [0x1B, 0x33]
    assert np.array_equal(vals, np.concatenate([np.full(16, 0.515625), np.full(16, 4.125)]))


def test_q4_error_bound():
    """Random blocks: every element is within half an E2M1 step (times the
    scale) of its input, or saturated at 6 * scale."""
    rng = np.random.default_rng(1)
    x = rng.normal(size=(64, 256)).astype(np.float32)
    codes, sc, vals = F.q4(x)
    d = np.repeat(F.e4m3_decode(sc), 16, axis=-1)
    err = np.abs(vals - x)
    ax = np.abs(x) / d
    # largest spacing between neighbours up to 6 is 2 (4 -> 6)
    half_step = np.where(ax < 2, 0.25, np.where(ax < 4, 0.5, 1.0)) * d
    sat = ax > 6
    assert np.all(err[~sat] <= half_step[~sat] * (1 + 1e-6))
    assert np.all(np.abs(vals[sat]) == 6 * d[sat])
