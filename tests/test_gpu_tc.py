"""The block-scaled NVFP4 tensor-core tile (tcgen05 kind::mxf4nvf4) against
the oracle's NVFP4 decode and a float64 product.

msk_debug_fp4_gemm multiplies one M = 128 x N = 16 tile through the same
shared-memory operand layouts, scale-factor chunks and MMA sequence as the
expert GEMMs of the layer kernel.  Checked here:

* exactness: with scales that keep every partial sum on a grid fp32 holds
  exactly (A scales 1, B scales in {1/2, 1, 2}: every product is a multiple
  of 1/8 and every sum stays below 2^21 of them), the result must equal the
  float64 product bit for bit, whatever the accumulation order;
* every E4M3 scale code on both operands, random codes: within the fp32
  accumulation bound K * 2^-23 * (|A| |B|^T) elementwise;
* single-element probes: B holding one 1.0 at (n, k) must give column n =
  A's column k and zeros elsewhere (pins the K and N placement).

Format: E2M1 elements with an E4M3 scale per 16 (the expert weights' NVFP4,
[newruntime] "What happened"; the W4A4 activations of the expert GEMMs,
[orcarouter] "Dove si colloca il confine del kernel")."""

import os

import numpy as np
import pytest
import torch

from oracle import formats as F

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_decode_step_persistent_gb300 as mod
    mod.load_library()
    return mod


def _dump(name, **arrays):
    d = os.environ.get("MSK_TEST_DUMP")
    if d:
        os.makedirs(d, exist_ok=True)
        np.savez(os.path.join(d, f"{name}.npz"), **arrays)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_tile(M, ac, as_, bc, bs):
    d = torch.full((128, 16), float("nan"), dtype=torch.float32, device="cuda")
    st = M.msk_debug_fp4_gemm(_dev(ac), _dev(as_), _dev(bc), _dev(bs), d)
    torch.cuda.synchronize()
    assert st == M.MSK_OK, f"msk_debug_fp4_gemm status {st}"
    return d.cpu().numpy().astype(np.float64)


def reference(ac, as_, bc, bs, K):
    A = F.nvfp4_dequant(ac, as_, 1.0, K)
    B = F.nvfp4_dequant(bc, bs, 1.0, K)
    ref = np.zeros((128, 16))
    ref[:, : B.shape[0]] = A @ B.T
    bound = np.zeros((128, 16))
    bound[:, : B.shape[0]] = np.abs(A) @ np.abs(B).T * K * 2.0 ** -23
    return ref, bound


def random_operand(rng, rows, K, scale_codes):
    codes = rng.integers(0, 16, size=(rows, K), dtype=np.uint8)
    return F.pack_nibbles(codes), rng.choice(np.asarray(scale_codes, dtype=np.uint8), size=(rows, K // 16))


@pytest.mark.parametrize("K,nb", [(2048, 16), (1024, 16), (128, 5), (384, 16)])
def test_tile_exact(M, K, nb):
    rng = np.random.default_rng(K + nb)
    ac, as_ = random_operand(rng, 128, K, [0x38])
    bc, bs = random_operand(rng, nb, K, [0x30, 0x38, 0x40])
    got = run_tile(M, ac, as_, bc, bs)
    ref, _ = reference(ac, as_, bc, bs, K)
    _dump(f"tile_exact_{K}_{nb}", ac=ac, as_=as_, bc=bc, bs=bs, got=got, ref=ref)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} elements differ, first {bad[:5].tolist()}: got {got[tuple(bad[0])]} " \
                          f"want {ref[tuple(bad[0])]}"


@pytest.mark.parametrize("K", [2048, 1024])
def test_tile_every_scale_code(M, K):
    rng = np.random.default_rng(7 + K)
    ac, as_ = random_operand(rng, 128, K, range(0x7F))
    bc, bs = random_operand(rng, 16, K, range(0x7F))
    as_.reshape(-1)[:127] = np.arange(127)
    bs.reshape(-1)[:127] = np.arange(127)
    got = run_tile(M, ac, as_, bc, bs)
    ref, bound = reference(ac, as_, bc, bs, K)
    _dump(f"tile_scales_{K}", ac=ac, as_=as_, bc=bc, bs=bs, got=got, ref=ref)
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"max excess {np.max(err - bound):.3e} at {np.unravel_index(np.argmax(err - bound), err.shape)}"


def test_tile_single_element_probes(M):
    """One 1.0 in B at (n, k) selects A's column k into D's column n."""
    K = 512
    rng = np.random.default_rng(3)
    ac, as_ = random_operand(rng, 128, K, range(0x28, 0x48))
    A = F.nvfp4_dequant(ac, as_, 1.0, K)
    for n, k in [(0, 0), (1, 1), (7, 31), (8, 32), (15, 63), (3, 64), (9, 255), (12, 256), (5, 300), (14, 511)]:
        codes = np.zeros((16, K), dtype=np.uint8)
        codes[n, k] = 2  # 1.0
        bc = F.pack_nibbles(codes)
        bs = np.full((16, K // 16), 0x38, dtype=np.uint8)
        got = run_tile(M, ac, as_, bc, bs)
        want = np.zeros((128, 16))
        want[:, n] = A[:, k]
        if not np.array_equal(got, want):
            nz = np.argwhere(got != 0)
            cols = sorted(set(nz[:, 1].tolist()))
            # which column of A does D's column n hold, if any
            match = [kk for kk in range(K) if np.array_equal(got[:, n], A[:, kk])]
            _dump(f"probe_{n}_{k}", ac=ac, as_=as_, got=got)
            pytest.fail(f"probe (n={n}, k={k}): nonzero D columns {cols}; D[:, {n}] equals A[:, {match[:4]}]")
