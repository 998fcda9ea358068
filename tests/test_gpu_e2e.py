"""Unforced end-to-end error of the verify step against the oracle.

The stage-by-stage checks (tests/test_gpu_parity.py) grade every stage on
the GPU's own inputs to it.  Here the oracle runs the whole step from the
step's input alone (hidden state and cache), and every layer's h2 and the
K/V rows each launch writes are compared with the GPU's, layer by layer:
max|err|/RMS(ref) and cosine, printed per layer.

The fp4 quantisers make a layer a discontinuous function of its input
(activation codes, intermediate codes and the top-k choice are rounding
decisions): ulp-level differences between fp32 accumulation on the GPU and
float64 in the oracle flip codes, and the flips compound from layer to
layer.  So the unforced bound is stated against the oracle's own
sensitivity: the oracle is run a second time from the same input with one
bf16 ulp added to 1% of its elements, and at every layer the GPU's
divergence from the oracle must stay within a few times the oracle's
divergence from itself (or within the stated 2e-2 * RMS, whichever is
larger), with cosine within a few times the oracle's own cosine loss of 1.
"""

import numpy as np
import pytest
import torch

import msk_synth as S
from oracle import model as OM
from tests._gpu import Setup, lt_to, run_layers, split_kv
from tests._util import np64, oracle_dims, oracle_weights, rel_stats

pytestmark = pytest.mark.gpu

SELF_FACTOR = 4.0   # GPU divergence allowed, in units of the oracle's self-divergence
FLOOR = 2e-2        # max|err| <= 2e-2 * RMS always passes
# Measured (stack8, current kernels): the GPU's divergence per layer is
# 0.5-1.1x the oracle's own divergence under the perturbation, for h2 and for
# the K / V rows; SELF_FACTOR leaves room for the step-to-step spread of
# that ratio.


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_decode_step_persistent_gb300 as M
    M.load_library()


def perturb_one_ulp(h: torch.Tensor, frac=0.01, seed=0) -> torch.Tensor:
    """h (bf16) with one bf16 ulp added to the magnitude of a seeded `frac`
    of its elements."""
    g = torch.Generator().manual_seed(seed)
    bits = h.detach().cpu().contiguous().view(torch.int16).clone()
    sel = torch.rand(bits.shape, generator=g) < frac
    bits[sel] += 1  # next bf16 away from zero (same sign)
    return bits.view(torch.bfloat16)


def oracle_unforced(dims, weights_of, windows, h0, caches, positions):
    """The oracle's step from h0 and the given caches (modified in place),
    launch by launch; weights_of(l) gives layer l's oracle weights.
    Returns per-layer h2 and the rows each launch wrote into the next
    layer's cache (the prologue's for layer 0)."""
    L = len(windows)
    w = weights_of(0)
    q, kr, vr = OM.qkv_project(dims, w, h0, positions)
    OM.write_kv(caches[0][0], caches[0][1], kr, vr, positions)
    rows = {0: (kr, vr)}
    h, h2s = h0, []
    for l in range(L):
        wn = weights_of(l + 1) if l + 1 < L else None
        Kn, Vn = caches[l + 1] if l + 1 < L else (None, None)
        o = OM.launch(dims, w, wn, q, h, caches[l][0], caches[l][1], positions, windows[l], Kn, Vn)
        h = o["h2"]
        h2s.append(h)
        if wn is not None:
            q = o["q_next"]
            rows[l + 1] = (o["k_next"], o["v_next"])
        w = wn
    return h2s, rows


def oracle_unforced_pair(dims, weights_of, windows, h0a, h0b, caches_a, caches_b, positions):
    """oracle_unforced from two inputs, launch by launch in lockstep (each
    layer's weights are fetched once for both)."""
    L = len(windows)
    w = weights_of(0)
    st = []
    for h0, caches in ((h0a, caches_a), (h0b, caches_b)):
        q, kr, vr = OM.qkv_project(dims, w, h0, positions)
        OM.write_kv(caches[0][0], caches[0][1], kr, vr, positions)
        st.append(dict(h=h0, q=q, caches=caches, h2s=[], rows={0: (kr, vr)}))
    for l in range(L):
        wn = weights_of(l + 1) if l + 1 < L else None
        for x in st:
            Kn, Vn = x["caches"][l + 1] if l + 1 < L else (None, None)
            o = OM.launch(dims, w, wn, x["q"], x["h"], x["caches"][l][0], x["caches"][l][1], positions, windows[l],
                          Kn, Vn)
            x["h"] = o["h2"]
            x["h2s"].append(o["h2"])
            if wn is not None:
                x["q"] = o["q_next"]
                x["rows"][l + 1] = (o["k_next"], o["v_next"])
        w = wn
    return st[0]["h2s"], st[0]["rows"], st[1]["h2s"], st[1]["rows"]


def gpu_rows(kv_l, positions):
    p = torch.tensor(positions, device=kv_l.device)
    k = kv_l[0][:, p, :].permute(1, 0, 2)
    v = kv_l[1][:, p, :].permute(1, 0, 2)
    return np64(k), np64(v)


def report(label, gpu_h2, gpu_kv, ref_h2, ref_rows, self_h2, self_rows):
    """Per-layer statistics, each (max|err|/RMS(ref), cosine), of the GPU's
    h2 and written K / V rows against the oracle, and of the perturbed
    oracle's against the oracle (the envelope)."""
    out = []
    for l in range(len(ref_h2)):
        g = (rel_stats(gpu_h2[l], ref_h2[l]), rel_stats(gpu_kv[l][0], ref_rows[l][0]),
             rel_stats(gpu_kv[l][1], ref_rows[l][1]))
        o = (rel_stats(self_h2[l], ref_h2[l]), rel_stats(self_rows[l][0], ref_rows[l][0]),
             rel_stats(self_rows[l][1], ref_rows[l][1]))
        out.append((l, g, o))
        print(f"{label} layer {l:2d}: GPU h2 {g[0][0]:.3e} {g[0][1]:.6f} K {g[1][0]:.3e} {g[1][1]:.6f} "
              f"V {g[2][0]:.3e} {g[2][1]:.6f} | oracle self h2 {o[0][0]:.3e} {o[0][1]:.6f} "
              f"K {o[1][0]:.3e} {o[1][1]:.6f} V {o[2][0]:.3e} {o[2][1]:.6f}")
    return out


def check_envelope(rep):
    """Every tensor of every layer: the GPU's max|err|/RMS within
    SELF_FACTOR times the oracle's own (or FLOOR), its 1 - cosine within
    SELF_FACTOR times the oracle's own (or 1e-3)."""
    for l, g, o in rep:
        for name, (e, c), (se, sc) in zip(("h2", "K rows", "V rows"), g, o):
            assert e <= max(FLOOR, SELF_FACTOR * se), f"layer {l} {name}: max|err|/rms {e:.3e}, oracle self {se:.3e}"
            assert 1 - c <= max(1e-3, SELF_FACTOR * (1 - sc)), f"layer {l} {name}: cosine {c:.6f}, oracle self {sc:.6f}"


def test_stack8_unforced_end_to_end():
    """The 8-layer stack (sliding x3, global) x2 over 8192 cached tokens."""
    wl = S.WORKLOADS["stack8"]
    st = Setup(wl, gen_device="cuda")
    kv = st.fresh_kv()
    kv_in = kv.clone()
    h0 = st.hidden()
    recs = run_layers(st, h0.clone(), kv, wl.positions, capture=False)
    torch.cuda.synchronize()
    gpu_h2 = [np64(r["h_out"]) for r in recs]
    gpu_kv = [gpu_rows(kv[l], wl.positions) for l in range(wl.n_layers)]
    caches = [split_kv(kv_in[l]) for l in range(wl.n_layers)]
    del kv, kv_in
    ref_h2, ref_rows = oracle_unforced(st.dims, st.ow, wl.windows, np64(h0), [tuple(c.copy() for c in kvp) for kvp in caches],
                                       wl.positions)
    self_h2, self_rows = oracle_unforced(st.dims, st.ow, wl.windows, np64(perturb_one_ulp(h0)), caches, wl.positions)
    check_envelope(report("stack8", gpu_h2, gpu_kv, ref_h2, ref_rows, self_h2, self_rows))
    st.model.close()


def test_full62_unforced_end_to_end():
    """The full 62-layer step (bench workload) against the oracle run on the
    host cores from the same input, and against the perturbed oracle for the
    envelope (both oracle runs in lockstep, layer weights regenerated one
    layer at a time: 62 layers do not fit the host as float64)."""
    from moe_decode_step_persistent_gb300 import Model
    wl = S.WORKLOADS["full62"]
    dims = oracle_dims(wl)
    model = Model(wl)
    for l in range(wl.n_layers):
        lt = S.layer_weights(wl, l, device="cuda")
        model.load_layer(l, lt)
        del lt
    torch.cuda.empty_cache()
    kv = torch.empty((wl.n_layers, 2, wl.n_kv_heads, wl.max_seq, wl.head_dim), dtype=torch.bfloat16, device="cuda")
    for l in range(wl.n_layers):
        S.fill_kv_cache(wl, l, kv[l])
    h0 = S.hidden_state(wl, device="cuda")
    h = h0.clone()
    gpu_h2 = []
    for l in range(wl.n_layers):
        model.layer_step(l, h, kv, wl.positions, run_prologue=(l == 0))
        gpu_h2.append(np64(h))
    gpu_kv = [gpu_rows(kv[l], wl.positions) for l in range(wl.n_layers)]
    del kv
    model.close()
    torch.cuda.empty_cache()

    cache_w = {}

    def weights_of(l):
        if l not in cache_w:
            for k in [k for k in cache_w if k < l - 1]:
                del cache_w[k]
            lt = S.layer_weights(wl, l, device="cuda")
            cache_w[l] = oracle_weights(lt_to(lt, "cpu"), wl)
            del lt
        return cache_w[l]

    class Caches:  # a layer's cache regenerated on demand (the oracle writes the verify rows)
        def __init__(self):
            self.c = {}

        def __getitem__(self, l):
            if l not in self.c:
                for k in [k for k in self.c if k < l - 1]:
                    del self.c[k]
                t = torch.empty((2, wl.n_kv_heads, wl.max_seq, wl.head_dim), dtype=torch.bfloat16, device="cuda")
                S.fill_kv_cache(wl, l, t)  # the same seeded stream the GPU run's cache came from
                self.c[l] = split_kv(t)
                del t
            return self.c[l]

    ref_h2, ref_rows, self_h2, self_rows = oracle_unforced_pair(
        dims, weights_of, wl.windows, np64(h0), np64(perturb_one_ulp(h0)), Caches(), Caches(), wl.positions)
    check_envelope(report("full62", gpu_h2, gpu_kv, ref_h2, ref_rows, self_h2, self_rows))
