"""Pins of the oracle's layer pieces: closed forms, brute force on tiny
shapes written independently of ``oracle.model`` (pure-Python loops over
keys / experts with math.fsum), and invariants.  No GPU."""

import math

import numpy as np
import pytest
import torch

import msk_synth as S
from oracle import formats as F
from oracle import model as OM
from tests._util import oracle_dims, oracle_weights, split_cache, np64


# ----------------------------------------------------------------------------
# RMSNorm
# ----------------------------------------------------------------------------


def test_rmsnorm_closed_forms():
    eps = 1e-6
    # constant row c: c / sqrt(c^2 + eps) -> 0.99999987.. -> bf16 1.0
    x = OM.rmsnorm(np.full((1, 4), 2.0), np.ones(4), eps)
    assert np.all(x == 1.0)
    # [3, 4, 0, 0]: mean square 6.25, rms 2.5 -> [1.2, 1.6, 0, 0];
    # bf16 neighbours of 1.2 are 1.1953125 / 1.203125 (nearer), of 1.6 are
    # 1.59375 / 1.6015625 (nearer)
    x = OM.rmsnorm(np.array([[3.0, 4.0, 0.0, 0.0]]), np.ones(4), eps)
    assert x.tolist() == [[1.203125, 1.6015625, 0.0, 0.0]]
    # gains multiply: gamma 2 on the 4 -> 3.2 -> bf16 3.203125
    x = OM.rmsnorm(np.array([[3.0, 4.0, 0.0, 0.0]]), np.array([1.0, 2.0, 1.0, 1.0]), eps)
    assert x[0, 1] == 3.203125
    # eps dominates a tiny row: 1e-4 / sqrt(1e-8 + 1e-6) = 0.0995.. (not 1.0)
    x = OM.rmsnorm(np.full((1, 2), 1e-4), np.ones(2), eps)
    assert abs(x[0, 0] - 1e-4 / math.sqrt(1e-8 + 1e-6)) < 1e-3


# ----------------------------------------------------------------------------
# RoPE
# ----------------------------------------------------------------------------


def test_rope_hand_cases():
    th = 1e6  # d=4: angles p * 1 and p * 1e-3
    e0 = np.array([[[1.0, 0.0, 0.0, 0.0]]])
    r = OM.rope(e0, [1], th)[0, 0]
    assert np.allclose(r, [math.cos(1), 0, math.sin(1), 0], atol=1e-15)
    e2 = np.array([[[0.0, 0.0, 1.0, 0.0]]])  # (a, b) = (0, 1) -> (-sin, cos)
    r = OM.rope(e2, [1], th)[0, 0]
    assert np.allclose(r, [-math.sin(1), 0, math.cos(1), 0], atol=1e-15)
    e1 = np.array([[[0.0, 1.0, 0.0, 0.0]]])  # second pair turns at 1e-3 rad/pos
    r = OM.rope(e1, [1000], th)[0, 0]
    assert np.allclose(r, [0, math.cos(1), 0, math.sin(1)], atol=1e-12)


def test_rope_invariants():
    rng = np.random.default_rng(0)
    v = rng.normal(size=(3, 2, 128))
    assert np.array_equal(OM.rope(v, [0, 0, 0], 1e6), v)  # p = 0 is the identity
    r = OM.rope(v, [5, 77, 16399], 1e6)
    half = 64
    n0 = v[..., :half] ** 2 + v[..., half:] ** 2
    n1 = r[..., :half] ** 2 + r[..., half:] ** 2
    assert np.allclose(n0, n1)  # every pair keeps its norm
    # q(p).k(p') depends only on p - p'
    q, k = rng.normal(size=(1, 1, 128)), rng.normal(size=(1, 1, 128))
    a = (OM.rope(q, [100], 1e6) * OM.rope(k, [90], 1e6)).sum()
    b = (OM.rope(q, [16010], 1e6) * OM.rope(k, [16000], 1e6)).sum()
    assert abs(a - b) < 1e-9


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------


def brute_attention(q, K, V, positions, window, G):
    T, Hq, d = q.shape
    out = np.zeros((T, Hq, d))
    for t in range(T):
        p = positions[t]
        keys = [j for j in range(p + 1) if window == 0 or j > p - window]
        for h in range(Hq):
            kv = h // G
            logits = [math.fsum(q[t, h, i] * K[kv, j, i] for i in range(d)) / math.sqrt(d) for j in keys]
            mx = max(logits)
            lse = mx + math.log(math.fsum(math.exp(l - mx) for l in logits))
            for i in range(d):
                out[t, h, i] = math.fsum(math.exp(l - lse) * V[kv, j, i] for l, j in zip(logits, keys))
    return out.reshape(T, -1)


@pytest.mark.parametrize("window", [0, 4, 7])
def test_attention_brute_force(window):
    rng = np.random.default_rng(window)
    dims = OM.Dims(hidden=16, n_q_heads=4, n_kv_heads=2, head_dim=8, pooled=8, n_experts=4,
                   top_k=2, inter=16)
    S_, T = 10, 3
    pos = [S_ + t for t in range(T)]
    q = F.rb(rng.normal(size=(T, 4, 8)))
    K = F.rb(rng.normal(size=(2, S_ + T, 8)))
    V = F.rb(rng.normal(size=(2, S_ + T, 8)))
    got = OM.attention(dims, q, K, V, pos, window)
    want = brute_attention(q, K, V, pos, window, G=2)
    # bf16 outputs: within half a bf16 step of the exact value
    assert np.all(np.abs(got - want) <= np.abs(want) * 2 ** -8 + 1e-300)


def test_attention_special_cases():
    dims = OM.Dims(hidden=8, n_q_heads=2, n_kv_heads=1, head_dim=4, pooled=8, n_experts=4,
                   top_k=1, inter=16)
    rng = np.random.default_rng(3)
    K = F.rb(rng.normal(size=(1, 6, 4)))
    V = F.rb(rng.normal(size=(1, 6, 4)))
    q = F.rb(rng.normal(size=(1, 2, 4)))
    # one visible key (position 0) -> output is V[0]
    o = OM.attention(dims, q, K, V, [0], 0).reshape(2, 4)
    assert np.array_equal(o[0], V[0, 0]) and np.array_equal(o[1], V[0, 0])
    # window 1 -> only the token itself
    o = OM.attention(dims, q, K, V, [4], 1).reshape(2, 4)
    assert np.array_equal(o[0], V[0, 4])
    # equal keys -> plain mean of the visible values
    K2 = np.ones_like(K)
    o = OM.attention(dims, q, K2, V, [5], 3).reshape(2, 4)
    assert np.allclose(o[0], V[0, 3:6].mean(axis=0), rtol=2 ** -8, atol=1e-12)


def test_attention_window_count():
    """A sliding layer sees exactly min(p + 1, W) keys: changing the key just
    outside the window changes nothing, the one just inside does."""
    dims = OM.Dims(hidden=8, n_q_heads=1, n_kv_heads=1, head_dim=4, pooled=8, n_experts=4,
                   top_k=1, inter=16)
    rng = np.random.default_rng(5)
    W, p = 6, 20
    K = F.rb(rng.normal(size=(1, 32, 4)))
    V = F.rb(rng.normal(size=(1, 32, 4)))
    q = F.rb(rng.normal(size=(1, 1, 4)))
    base = OM.attention(dims, q, K, V, [p], W)
    K_out, V_out = K.copy(), V.copy()
    K_out[0, p - W] += 5
    V_out[0, p - W] += 5
    assert np.array_equal(OM.attention(dims, q, K_out, V_out, [p], W), base)
    V_in = V.copy()
    V_in[0, p - W + 1] += 5
    assert not np.array_equal(OM.attention(dims, q, K, V_in, [p], W), base)
    assert OM.visible_range(p, W) == (p - W + 1, p)
    assert OM.visible_range(3, 2048) == (0, 3) and OM.visible_range(5000, 0) == (0, 5000)
    # 2048-window at p >= 2047 masks all but exactly 2048 positions
    lo, hi = OM.visible_range(4096 + 7, 2048)
    assert hi - lo + 1 == 2048


# ----------------------------------------------------------------------------
# router
# ----------------------------------------------------------------------------


def _router_setup(E, k, logits_row):
    dims = OM.Dims(hidden=8, n_q_heads=1, n_kv_heads=1, head_dim=4, pooled=E, n_experts=E,
                   top_k=k, inter=16)
    # pooled = identity rows so that logits = the given values exactly
    w = OM.LayerWeights(attn_norm=None, moe_norm=None, w_qkv=None, w_o=None, w_pool=None,
                        w_router=np.eye(E), router_bias=np.zeros(E), w_unpool=None)
    pooled = np.asarray(logits_row, dtype=np.float64)[None, :]
    return dims, w, pooled


def test_topk_ties_and_order():
    dims, w, pooled = _router_setup(6, 3, [1.0, 3.0, 2.0, 3.0, 2.0, 0.5])
    idx, gates, _ = OM.router(dims, w, pooled)
    assert idx.tolist() == [[1, 3, 2]]  # 3.0 (lower index first), then 2.0 at index 2
    e = np.exp([0.0, 0.0, -1.0])
    assert np.allclose(gates[0], e / e.sum())


def test_topk_brute_force_and_bias():
    rng = np.random.default_rng(7)
    E, k, T = 16, 4, 5
    dims = OM.Dims(hidden=8, n_q_heads=1, n_kv_heads=1, head_dim=4, pooled=8, n_experts=E,
                   top_k=k, inter=16)
    w = OM.LayerWeights(attn_norm=None, moe_norm=None, w_qkv=None, w_o=None, w_pool=None,
                        w_router=F.rb(rng.normal(size=(E, 8))),
                        router_bias=F.f32(rng.normal(size=E)), w_unpool=None)
    pooled = F.rb(rng.normal(size=(T, 8)))
    idx, gates, logits = OM.router(dims, w, pooled)
    for t in range(T):
        raw = [math.fsum(pooled[t, i] * w.w_router[e, i] for i in range(8)) for e in range(E)]
        lg = [float(np.float32(np.float32(raw[e]) + np.float32(w.router_bias[e]))) for e in range(E)]
        order = sorted(range(E), key=lambda e: (-lg[e], e))[:k]
        assert idx[t].tolist() == order
        ex = [math.exp(lg[e] - lg[order[0]]) for e in order]
        assert np.allclose(gates[t], np.array(ex) / math.fsum(ex), rtol=1e-12)
        assert abs(gates[t].sum() - 1.0) < 1e-12


def test_topk_k1_gate_is_one():
    dims, w, pooled = _router_setup(5, 1, [0.1, 0.7, -2.0, 0.69, 0.0])
    idx, gates, _ = OM.router(dims, w, pooled)
    assert idx.tolist() == [[1]] and gates.tolist() == [[1.0]]


def test_silu():
    assert OM.silu(np.array(0.0)) == 0.0
    assert abs(OM.silu(np.array(40.0)) - 40.0) < 1e-12
    assert abs(OM.silu(np.array(-40.0))) < 1e-15
    x = np.array(1.3)
    assert abs(OM.silu(x) - OM.silu(-x) - x) < 1e-15  # silu(x) - silu(-x) = x


# ----------------------------------------------------------------------------
# experts: independent per-element path
# ----------------------------------------------------------------------------

E2M1 = [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def _e2m1(c):
    return -E2M1[c & 7] if c & 8 else E2M1[c & 7]


def _e4m3(b):
    s, e, m = b >> 7, (b >> 3) & 15, b & 7
    v = (m / 8) * 2 ** -6 if e == 0 else (1 + m / 8) * 2 ** (e - 7)
    return -v if s else v


def _w(ex, r, c):
    byte = int(ex.packed[r, c // 2])
    code = byte & 15 if c % 2 == 0 else byte >> 4
    return float(np.float32(np.float32(_e2m1(code) * _e4m3(int(ex.scales[r, c // 16]))) * np.float32(ex.tensor_scale)))


def test_expert_brute_force():
    wl = S.scaled(S.WORKLOADS["tiny"], hidden=32, pooled=32, inter=32, n_experts=4, top_k=2,
                  n_q_heads=2, n_kv_heads=1, head_dim=16)
    lt = S.layer_weights(wl, 0)
    w = oracle_weights(lt, wl)
    dims = oracle_dims(wl)
    rng = np.random.default_rng(11)
    pooled = F.rb(rng.normal(size=(2, 32)) * 1.3)
    idx = np.array([[2, 0], [1, 2]])
    gates = np.array([[0.7, 0.3], [0.55, 0.45]])
    m, y, _ = OM.experts(dims, w, pooled, idx, gates)
    for t in range(2):
        a = F.q4(pooled[t])[2]
        ys = []
        for r in range(2):
            e = idx[t, r]
            g = [math.fsum(_w(w.gate[e], i, c) * a[c] for c in range(32)) for i in range(32)]
            u = [math.fsum(_w(w.up[e], i, c) * a[c] for c in range(32)) for i in range(32)]
            s = np.array([gi / (1 + math.exp(-gi)) * ui for gi, ui in zip(g, u)], dtype=np.float32)
            sq = F.q4(s.astype(np.float64))[2]
            yv = F.rb(np.array([math.fsum(_w(w.down[e], p, c) * sq[c] for c in range(32)) for p in range(32)]))
            assert np.allclose(yv, y[t, r], rtol=2 ** -7, atol=1e-30)
            ys.append(yv)
        mm = F.rb(gates[t, 0] * ys[0] + gates[t, 1] * ys[1])
        assert np.allclose(mm, m[t], rtol=2 ** -7, atol=1e-30)


# ----------------------------------------------------------------------------
# whole-layer invariants on the tiny workload
# ----------------------------------------------------------------------------


def _tiny_layer(tokens=1, cached=128, window=0, gamma_std=0.0, layers=1):
    wl = S.scaled(S.WORKLOADS["tiny"], tokens=tokens, cached=cached, windows=(window,) * layers)
    lts = [S.layer_weights(wl, l, gamma_std=gamma_std) for l in range(layers)]
    ws = [oracle_weights(lt, wl) for lt in lts]
    caches = [split_cache(S.kv_cache(wl, l)) for l in range(layers)]
    h = np64(S.hidden_state(wl))
    return wl, oracle_dims(wl), ws, caches, h


def test_layer_zero_projections_pass_residual():
    wl, dims, ws, caches, h = _tiny_layer(tokens=2)
    w = ws[0]
    K, V = caches[0]
    q, kr, vr = OM.qkv_project(dims, w, h, wl.positions)
    OM.write_kv(K, V, kr, vr, wl.positions)
    w.w_o = np.zeros_like(w.w_o)
    for ex in w.down:
        ex.packed = np.zeros_like(ex.packed)
    out = OM.launch(dims, w, None, q, h, K, V, wl.positions, 0)
    assert np.array_equal(out["h1"], h)
    assert np.array_equal(out["h2"], out["h1"])
    assert np.all(out["m"] == 0)


def test_layer_expert_permutation_invariance():
    wl, dims, ws, caches, h = _tiny_layer(tokens=2, gamma_std=0.1)
    w = ws[0]
    K, V = caches[0]
    q, kr, vr = OM.qkv_project(dims, w, h, wl.positions)
    OM.write_kv(K, V, kr, vr, wl.positions)
    base = OM.launch(dims, w, None, q, h, K, V, wl.positions, 0)
    perm = np.random.default_rng(2).permutation(dims.n_experts)
    w.w_router = w.w_router[perm]
    w.router_bias = w.router_bias[perm]
    w.gate = [w.gate[i] for i in perm]
    w.up = [w.up[i] for i in perm]
    w.down = [w.down[i] for i in perm]
    out = OM.launch(dims, w, None, q, h, K, V, wl.positions, 0)
    assert np.array_equal(out["h2"], base["h2"])
    assert np.array_equal(perm[out["idx"]], base["idx"]) or np.all(
        np.sort(perm[out["idx"]], 1) == np.sort(base["idx"], 1))


def test_decode_step_causal_prefix():
    """Perturbing token t's input changes no output of tokens < t."""
    wl, dims, ws, caches, h = _tiny_layer(tokens=3, cached=40, window=16, layers=2)
    c1 = [(K.copy(), V.copy()) for K, V in caches]
    hA, _ = OM.decode_step(dims, ws, wl.windows, h, c1, wl.positions)
    h2 = h.copy()
    h2[2] += 0.5
    c2 = [(K.copy(), V.copy()) for K, V in caches]
    hB, _ = OM.decode_step(dims, ws, wl.windows, h2, c2, wl.positions)
    assert np.array_equal(hA[:2], hB[:2])
    assert not np.array_equal(hA[2], hB[2])


def test_decode_step_chains_launches():
    """The step equals prologue + one launch per layer with each launch
    writing the next layer's KV rows."""
    wl, dims, ws, caches, h = _tiny_layer(tokens=2, cached=24, window=8, layers=3)
    ca = [(K.copy(), V.copy()) for K, V in caches]
    hA, outs = OM.decode_step(dims, ws, wl.windows, h, ca, wl.positions)
    cb = [(K.copy(), V.copy()) for K, V in caches]
    q, kr, vr = OM.qkv_project(dims, ws[0], h, wl.positions)
    OM.write_kv(cb[0][0], cb[0][1], kr, vr, wl.positions)
    x = h
    for l in range(3):
        o = OM.launch(dims, ws[l], None, q, x, cb[l][0], cb[l][1], wl.positions, wl.windows[l])
        x = o["h2"]
        if l < 2:
            q, kr, vr = OM.qkv_project(dims, ws[l + 1], x, wl.positions)
            OM.write_kv(cb[l + 1][0], cb[l + 1][1], kr, vr, wl.positions)
    assert np.array_equal(hA, x)
    for l in range(3):
        assert np.array_equal(ca[l][0], cb[l][0]) and np.array_equal(ca[l][1], cb[l][1])
