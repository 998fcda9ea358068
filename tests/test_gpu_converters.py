"""The kernel's E2M1 and E4M3 conversions (round to nearest, ties to even,
saturating; the activation quantiser's building blocks) against the oracle's
converters, over EVERY fp32 value whose conversion is not trivially zero or
saturated: all 2^23 mantissas of every exponent from 2^-12 to 2^9 (E4M3's
smallest subnormal is 2^-9, its largest value 448; E2M1's are 0.5 and 6),
for positive values, with negative values checked by sign symmetry on the
GPU; plus subnormals, zeros, huge values and infinities by sample.  Codes
must match exactly; a value that rounds to zero may carry either sign."""

import numpy as np
import pytest
import torch

from oracle import formats as F

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_decode_step_persistent_gb300 as M
    M.load_library()  # raises if the extension is missing: no fallback


def _gpu_codes(x_gpu):
    import moe_decode_step_persistent_gb300 as M
    e2 = torch.empty(x_gpu.shape, dtype=torch.uint8, device="cuda")
    e4 = torch.empty(x_gpu.shape, dtype=torch.uint8, device="cuda")
    M.msk_debug_convert(x_gpu, e2, e4)
    return e2, e4


def _check(xs_cpu, e2, e4):
    x64 = xs_cpu.numpy().astype(np.float64)
    want2 = F.e2m1_encode_rn(x64)
    want4 = F.e4m3_encode_rn(x64)
    got2, got4 = e2.cpu().numpy(), e4.cpu().numpy()
    # a value that rounds to zero: either sign of zero
    z2 = (want2 & 7) == 0
    z4 = (want4 & 0x7F) == 0
    bad2 = np.where(z2, (got2 & 7) != 0, got2 != want2)
    bad4 = np.where(z4, (got4 & 0x7F) != 0, got4 != want4)
    assert not bad2.any(), f"E2M1: {bad2.sum()} mismatches, first x={x64[bad2][:4]} got {got2[bad2][:4]} want {want2[bad2][:4]}"
    assert not bad4.any(), f"E4M3: {bad4.sum()} mismatches, first x={x64[bad4][:4]} got {got4[bad4][:4]} want {want4[bad4][:4]}"


def test_every_fp32_value_in_the_converters_range():
    mant = torch.arange(1 << 23, dtype=torch.int32, device="cuda")
    for e in range(-12, 10):
        bits = mant | ((e + 127) << 23)
        x = bits.view(torch.float32)
        e2, e4 = _gpu_codes(x)
        _check(x.cpu(), e2, e4)
        # negative values: the same codes with the sign bit (zero keeps either sign)
        n2, n4 = _gpu_codes(-x)
        nz2 = (e2 & 7) != 0
        nz4 = (e4 & 0x7F) != 0
        assert torch.equal(n2[nz2], e2[nz2] | 8), e
        assert torch.equal(n4[nz4], e4[nz4] | 0x80), e
        assert torch.all((n2[~nz2] & 7) == 0) and torch.all((n4[~nz4] & 0x7F) == 0), e


def test_specials_and_outside_the_range():
    rng = np.random.default_rng(0)
    sub = rng.integers(1, 1 << 23, size=4096, dtype=np.int64)  # subnormals
    tiny = (rng.integers(1, 115, size=4096) << 23) | rng.integers(0, 1 << 23, size=4096)  # 2^-126 .. 2^-13
    huge = ((rng.integers(137, 255, size=4096)) << 23) | rng.integers(0, 1 << 23, size=4096)  # 2^10 .. 2^127
    specials = np.array([0, 0x7F800000], dtype=np.int64)  # 0, +inf
    b = np.concatenate([sub, tiny, huge, specials]).astype(np.uint32)
    b = np.concatenate([b, b | 0x80000000]).view(np.int32)
    x = torch.from_numpy(b).view(torch.float32)
    e2, e4 = _gpu_codes(x.cuda())
    _check(x, e2, e4)
