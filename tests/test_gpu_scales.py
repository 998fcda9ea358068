"""GPU parity of the NVFP4 weight path over every E4M3 block-scale code.

The seeded generator draws block scales from a narrow code range; these
tests load experts whose scales run through every finite code 0x00..0x7E
(zero, all subnormals 2^-9..7*2^-9, up to 448) and the hand-built blocks of
tests/golden/nvfp4_blocks.txt, then check

* msk_debug_dequant (the library's repacked layout, read back) bit for bit
  against the oracle's NVFP4 decode and against the hand-written values;
* one launch whose routing uses only such experts, stage by stage against
  the oracle (the expert GEMMs see every scale code);
* that a block scale with the sign bit set, or the E4M3 NaN code, makes
  msk_load_layer return MSK_ERR_BAD_SCALE, and that a clean load and a
  launch still work afterwards.

Format source: expert weights in 4-bit NVFP4 ([newruntime] "What happened";
[orcarouter] "Dove si colloca il confine del kernel"); E2M1 elements with
an E4M3 scale per 16 and an fp32 tensor scale per matrix, per the workload
definition."""

import os

import numpy as np
import pytest
import torch

import msk_synth as S
from oracle import formats as F
from tests._gpu import Setup, check_launch, lt_to, run_layers
from tests._util import oracle_dims

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "nvfp4_blocks.txt")
MSK_ERR_BAD_SCALE = 4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_decode_step_persistent_gb300 as M
    M.load_library()


def golden_blocks():
    """(name, packed bytes [8], scale code, tensor scale, values [16])."""
    out = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#") or line.startswith("case"):
                continue
            r = line.split()
            packed = np.array([int(b, 16) for b in r[1].split(",")], dtype=np.uint8)
            out.append((r[0], packed, int(r[2], 16), float(r[3]), np.array([float(v) for v in r[4:]])))
    assert len(out) == 6
    return out


GOLD_EXPERT = -1  # the last expert holds the hand-built blocks and is never routed


def full_range(lt, wl):
    """Every matrix of every expert: block scale codes cycling through all
    finite codes 0x00..0x7E (each matrix holds >= 127 blocks).  The last
    expert gets the hand-built blocks (gate rows 0-3: blocks A-D, tensor
    scale 1; up rows 0-1: blocks E-F, tensor scale 0.3f) and a router bias
    that keeps it out of every top-k."""
    for m, trip in enumerate((lt.gate, lt.up, lt.down)):
        packed, scales, ts = trip
        E, rows, nb = scales.shape
        assert rows * nb >= 127
        i = torch.arange(rows * nb).reshape(rows, nb)
        for e in range(E):
            scales[e] = ((i + 17 * e + 41 * m) % 127).to(torch.uint8)
        if m < 2:
            # at this small width the SwiGLU outputs would otherwise fall below
            # the smallest E4M3 block scale and quantise to zero
            ts *= 64.0
    gb = golden_blocks()
    gp, gs, gts = lt.gate
    up, us, uts = lt.up
    for r, (_, packed, sc, ts, _) in enumerate(gb[:4]):
        assert ts == 1.0
        gp[GOLD_EXPERT, r, :8] = torch.from_numpy(packed)
        gs[GOLD_EXPERT, r, 0] = sc
    gts[GOLD_EXPERT] = 1.0
    for r, (_, packed, sc, ts, _) in enumerate(gb[4:]):
        up[GOLD_EXPERT, r, :8] = torch.from_numpy(packed)
        us[GOLD_EXPERT, r, 0] = sc
        uts[GOLD_EXPERT] = ts
    lt.router_bias[GOLD_EXPERT] = -1.0e4


class ScaleSetup(Setup):
    """Setup with the weights passed through `mutate` before loading."""

    def __init__(self, wl, mutate, gamma_std=0.0):
        from moe_decode_step_persistent_gb300 import Model
        self.wl = wl
        self.dims = oracle_dims(wl)
        self.model = Model(wl)
        self.lts_cpu = []
        for l in range(wl.n_layers):
            lt = S.layer_weights(wl, l, device="cpu", gamma_std=gamma_std)
            mutate(lt, wl)
            self.model.load_layer(l, lt_to(lt, "cuda"))
            self.lts_cpu.append(lt)
        torch.cuda.synchronize()
        self._ow = {}


def _wl():
    # 16 verify tokens, 16 experts top-2, pooled = inter = 128: every matrix
    # is 128 x 128 (1,024 blocks, each scale code 8 times)
    return S.scaled(S.WORKLOADS["tiny"], tokens=16, cached=64, windows=(0, 0))


def _dequant(st, layer, e, which):
    trip = (st.lts_cpu[layer].gate, st.lts_cpu[layer].up, st.lts_cpu[layer].down)[which]
    rows, cols = trip[0].shape[1], trip[0].shape[2] * 2
    out = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    st.model.debug_dequant(layer, e, which, out)
    ref = F.nvfp4_dequant(trip[0][e].numpy(), trip[1][e].numpy(), float(trip[2][e]), cols)
    return out.cpu().numpy().astype(np.float64), ref


def test_dequant_every_scale_code():
    wl = _wl()
    st = ScaleSetup(wl, full_range)
    seen = set()
    for e in range(wl.n_experts):
        for which in range(3):
            got, ref = _dequant(st, 0, e, which)
            assert np.array_equal(got, ref), (e, which)
            assert np.array_equal(np.signbit(got), np.signbit(ref)), (e, which)
            seen |= set((st.lts_cpu[0].gate, st.lts_cpu[0].up, st.lts_cpu[0].down)[which][1][e].flatten().tolist())
    assert seen == set(range(127))
    st.model.close()


def test_dequant_hand_built_blocks():
    """The GPU reads the six hand-built blocks back with exactly the values
    (and zero signs) written by hand in tests/golden/nvfp4_blocks.txt."""
    st = ScaleSetup(_wl(), full_range)
    e = st.wl.n_experts + GOLD_EXPERT
    gate, _ = _dequant(st, 0, e, 0)
    up, _ = _dequant(st, 0, e, 1)
    gb = golden_blocks()
    for r, (name, _, _, _, want) in enumerate(gb[:4]):
        assert np.array_equal(gate[r, :16], want), name
        assert np.array_equal(np.signbit(gate[r, :16]), np.signbit(want)), name
    for r, (name, _, _, _, want) in enumerate(gb[4:]):
        assert np.array_equal(up[r, :16], want), name
        assert np.array_equal(np.signbit(up[r, :16]), np.signbit(want)), name
    st.model.close()


def test_launch_with_every_scale_code():
    """Two launches whose experts carry every scale code: every stage against
    the oracle (teacher forced; see tests/_gpu.py)."""
    wl = _wl()
    st = ScaleSetup(wl, full_range, gamma_std=0.1)
    kv = st.fresh_kv()
    h = st.hidden()
    recs = run_layers(st, h, kv, wl.positions)
    torch.cuda.synchronize()
    rep = []
    for r in recs:
        check_launch(st, r, kv, wl.positions, rep)
        assert (st.wl.n_experts + GOLD_EXPERT) not in set(r["routing"].cpu().flatten().tolist())
        # the GEMMs saw real data: most fp4-intermediate blocks are nonzero
        assert (r["sq_scales"] != 0).float().mean().item() > 0.5
    for l, o in rep:
        print("every-scale-code launch", l, {k: o[k] for k in ("y", "m", "h2", "sq_match", "unique_experts")})
    st.model.close()


@pytest.mark.parametrize("code", [0x80, 0xB8, 0xFE, 0x7F, 0xFF])
def test_bad_scale_rejected(code):
    """Sign bit set (0x80 = -0, 0xB8 = -1, 0xFE = -448) or NaN (0x7F, 0xFF):
    MSK_ERR_BAD_SCALE, whichever matrix holds it; afterwards a clean load of
    the same layer and a launch succeed."""
    import moe_decode_step_persistent_gb300 as M
    wl = S.scaled(_wl(), windows=(0,))
    from moe_decode_step_persistent_gb300 import Model
    model = Model(wl)
    lt = S.layer_weights(wl, 0, device="cpu")
    for which, (e, r, b) in enumerate([(3, 5, 2), (0, 127, 7), (15, 64, 0)]):
        bad = S.LayerTensors(**{k: getattr(lt, k) for k in ("attn_norm", "moe_norm", "w_qkv", "w_o", "w_pool",
                                                              "w_router", "router_bias", "w_unpool")},
                             gate=tuple(x.clone() for x in lt.gate), up=tuple(x.clone() for x in lt.up),
                             down=tuple(x.clone() for x in lt.down))
        trip = (bad.gate, bad.up, bad.down)[which]
        trip[1][e, r, b] = code
        with pytest.raises(M.MskError) as ei:
            model.load_layer(0, lt_to(bad, "cuda"))
        assert ei.value.status == MSK_ERR_BAD_SCALE
    model.load_layer(0, lt_to(lt, "cuda"))
    kv = torch.zeros((1, 2, wl.n_kv_heads, wl.max_seq, wl.head_dim), dtype=torch.bfloat16, device="cuda")
    S.fill_kv_cache(wl, 0, kv[0])
    h = S.hidden_state(wl, device="cpu").to("cuda")
    model.layer_step(0, h, kv, wl.positions, run_prologue=True)
    assert torch.isfinite(h.float()).all()
    model.close()
