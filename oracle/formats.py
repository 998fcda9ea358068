"""Number formats of the verify step: bf16 storage, NVFP4 (E2M1 + E4M3).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The pages state that expert weights are stored in 4-bit NVFP4 while other
layers stay in bf16 ([newruntime] §What happened; [orcarouter] §Dove si
colloca il confine del kernel), and that the first expert GEMM's output
travels as fp4 and the second's as bf16 ([orcarouter] same section).  The
block layout is the workload's: E2M1 element codes, one E4M3 scale per 16
consecutive elements along K, and one fp32 tensor scale per matrix.

Everything here is written from the format definitions:
  * E2M1: sign bit 3, 2 exponent bits (bias 1), 1 mantissa bit; magnitudes
    0, 0.5, 1, 1.5, 2, 3, 4, 6; no inf/NaN.
  * E4M3 (the "FN" variant): sign bit 7, 4 exponent bits (bias 7), 3 mantissa
    bits; exponent 0 is subnormal (m/8)*2^-6; S.1111.111 is NaN; no inf;
    largest finite 448.
  * Round-to-nearest-even with saturation to the largest finite value
    ("satfinite"): the nearest representable magnitude; on an exact tie the
    code whose lowest bit is 0.
"""

from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------
# bf16 / fp32 storage rounding
# ----------------------------------------------------------------------------


def rb(x):
    """Round to the nearest bf16 value (ties to even), returned as float64.

    bf16 keeps 8 significant bits and fp32's exponent range.  Rounding is
    done directly from float64 (no detour through float32, which would round
    twice).  Values below the bf16 normal range round on the subnormal grid
    of spacing 2^-133.  Overflow goes to +-inf.  NaN stays NaN.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = np.isfinite(x) & (x != 0)
    v = x[nz]
    _, e = np.frexp(v)  # v = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)  # below 2^-126 the grid is fixed (subnormals)
    step = np.ldexp(1.0, e - 8)  # spacing of 8-significant-bit values
    r = np.rint(v / step) * step  # np.rint rounds half to even
    r[np.abs(r) > 3.3895313892515355e38] = np.inf * np.sign(r[np.abs(r) > 3.3895313892515355e38])
    out[nz] = r
    out[~np.isfinite(x)] = x[~np.isfinite(x)]
    return out


def f32(x):
    """Round to float32 (ties to even), returned as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# E2M1
# ----------------------------------------------------------------------------

#: magnitudes of E2M1 codes 0..7 (code 8..15 are the negatives)
E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_decode(codes):
    """Value of 4-bit E2M1 codes (uint8 0..15)."""
    codes = np.asarray(codes, dtype=np.int64)
    mag = E2M1_MAG[codes & 7]
    return np.where(codes & 8, -mag, mag)


# ----------------------------------------------------------------------------
# E4M3
# ----------------------------------------------------------------------------


def e4m3_decode(codes):
    """Value of 8-bit E4M3 codes (uint8 0..255); NaN for S.1111.111."""
    codes = np.asarray(codes, dtype=np.int64)
    s = (codes >> 7) & 1
    e = (codes >> 3) & 15
    m = codes & 7
    normal = (1.0 + m / 8.0) * np.ldexp(1.0, e - 7)
    sub = (m / 8.0) * np.ldexp(1.0, -6)
    mag = np.where(e == 0, sub, normal)
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


#: magnitudes of the finite non-negative E4M3 codes 0x00..0x7E, ascending
E4M3_MAG = e4m3_decode(np.arange(0x7F))


def _rn_even_code(x, mag_table):
    """Code of the nearest magnitude in ``mag_table`` (ascending, indexed by
    code) to |x|, ties to the even code, saturating at the last entry."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    hi = np.searchsorted(mag_table, ax, side="left")
    hi = np.clip(hi, 0, len(mag_table) - 1)
    lo = np.clip(hi - 1, 0, len(mag_table) - 1)
    d_hi = np.abs(mag_table[hi] - ax)
    d_lo = np.abs(ax - mag_table[lo])
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(pick_lo, lo, hi)
    # above the largest finite magnitude: saturate
    code = np.where(ax >= mag_table[-1], len(mag_table) - 1, code)
    return code.astype(np.int64)


def e2m1_encode_rn(x):
    """E2M1 code of float values, round-to-nearest-even, satfinite.

    The sign bit follows the sign of x (negative values that round to zero
    give code 8, i.e. -0)."""
    x = np.asarray(x, dtype=np.float64)
    code = _rn_even_code(x, E2M1_MAG)
    return np.where(np.signbit(x), code | 8, code).astype(np.uint8)


def e4m3_encode_rn(x):
    """E4M3 code of float values, round-to-nearest-even, satfinite.
    NaN maps to 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    code = _rn_even_code(np.nan_to_num(x), E4M3_MAG)
    code = np.where(np.signbit(x), code | 0x80, code)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


# ----------------------------------------------------------------------------
# NVFP4 tensors
# ----------------------------------------------------------------------------


def unpack_nibbles(packed, cols):
    """[rows][cols/2] bytes -> [rows][cols] codes; element 2i is the low
    nibble of byte i, element 2i+1 the high nibble."""
    packed = np.asarray(packed, dtype=np.uint8)
    lo = packed & 0x0F
    hi = packed >> 4
    out = np.empty(packed.shape[:-1] + (cols,), dtype=np.uint8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def pack_nibbles(codes):
    """Inverse of :func:`unpack_nibbles`."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] & 0x0F) | ((codes[..., 1::2] & 0x0F) << 4)


def nvfp4_dequant(packed, scales, tensor_scale, cols):
    """Dequantised NVFP4 matrix [rows][cols] as float64 values of float32s.

    w = fp32(e2m1 * e4m3) * tensor_scale, with the second product one fp32
    round-to-nearest-even multiply.  (e2m1 * e4m3 has at most 6 significant
    bits and is exact in fp32, so this is reproducible bit for bit.)

    packed: [rows][cols/2] uint8; scales: [rows][cols/16] uint8 E4M3 codes.
    """
    codes = unpack_nibbles(packed, cols)
    blk = np.repeat(e4m3_decode(scales), 16, axis=-1)
    prod = (e2m1_decode(codes) * blk).astype(np.float32)  # exact
    ts = np.float32(tensor_scale)
    return (prod * ts).astype(np.float32).astype(np.float64)


def q4(x, block=16):
    """Activation quantiser Q4 along the last axis, blocks of 16.

    Decisions are taken on float32 values with float32 arithmetic:
      amax = max |x| over the block;
      amax == 0             -> scale code 0, all element codes 0;
      sc   = E4M3_RN(fp32(amax / 6));  dec(sc) == 0 -> zero block;
      code = E2M1_RN(fp32(x / dec(sc))) for each element.
    The activation tensor scale is 1.

    Returns (codes uint8 [..., n], scale codes uint8 [..., n/16], values
    float64 [..., n] = e2m1 * e4m3 exactly).
    """
    x = np.asarray(x, dtype=np.float64).astype(np.float32)
    shp = x.shape
    xb = x.reshape(shp[:-1] + (shp[-1] // block, block))
    amax = np.max(np.abs(xb), axis=-1)
    sc = e4m3_encode_rn((amax / np.float32(6.0)).astype(np.float32))
    sc = np.where(amax == 0, 0, sc).astype(np.uint8)
    dsc = e4m3_decode(sc).astype(np.float32)
    zero_blk = dsc == 0
    safe = np.where(zero_blk, np.float32(1.0), dsc).astype(np.float32)
    ratio = (xb / safe[..., None]).astype(np.float32)
    codes = e2m1_encode_rn(ratio)
    codes = np.where(zero_blk[..., None], 0, codes).astype(np.uint8)
    vals = e2m1_decode(codes) * np.where(zero_blk, 0.0, dsc.astype(np.float64))[..., None]
    return codes.reshape(shp), sc, vals.reshape(shp)
