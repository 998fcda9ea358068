"""Pins of the oracle's tree-of-candidates verification ([orcarouter], the
draft section: the verified block is a tree of candidate tokens rather than
a linear chain).  Slot t has a parent slot (or -1 for a child of the
context); its position is the cached length plus its depth; it attends to
the context and to its ancestors and itself.  Brute force below is written
independently of ``oracle.model`` (parent walks and math.fsum loops).  No
GPU."""

import math

import numpy as np
import pytest

import msk_synth as S
from oracle import formats as F
from oracle import model as OM
from tests._util import np64, oracle_dims, oracle_weights, split_cache


def _depth(parents, t):
    d = 0
    while parents[t] >= 0:
        t = parents[t]
        d += 1
    return d


def _is_ancestor_or_self(parents, u, t):
    while t >= 0:
        if t == u:
            return True
        t = parents[t]
    return False


def brute_tree_attention(q, K, V, S_, parents, window, G):
    """Keys of slot t: cached rows j < S_ and verify rows S_ + u (u an
    ancestor of t or t itself); a key at position x is visible if
    window == 0 or x > p_t - window, with p_t = S_ + depth(t)."""
    T, Hq, d = q.shape
    out = np.zeros((T, Hq, d))
    for t in range(T):
        p = S_ + _depth(parents, t)
        keys = [j for j in range(S_) if window == 0 or j > p - window]
        keys += [S_ + u for u in range(T)
                 if _is_ancestor_or_self(parents, u, t) and (window == 0 or S_ + _depth(parents, u) > p - window)]
        for h in range(Hq):
            kv = h // G
            logits = [math.fsum(q[t, h, i] * K[kv, j, i] for i in range(d)) / math.sqrt(d) for j in keys]
            mx = max(logits)
            lse = mx + math.log(math.fsum(math.exp(x - mx) for x in logits))
            for i in range(d):
                out[t, h, i] = math.fsum(math.exp(x - lse) * V[kv, j, i] for x, j in zip(logits, keys))
    return out.reshape(T, -1)


def _dims():
    return OM.Dims(hidden=16, n_q_heads=4, n_kv_heads=2, head_dim=8, pooled=8, n_experts=4, top_k=2,
                   inter=16)


def test_tree_depths_and_ancestors_by_hand():
    #        ctx
    #       /    \
    #      0      4
    #     / \     |
    #    1   2    5
    #    |
    #    3
    par = [-1, 0, 0, 1, -1, 4]
    assert OM.tree_depths(par) == [0, 1, 1, 2, 0, 1]
    assert OM.tree_ancestors(par) == [[0], [0, 1], [0, 2], [0, 1, 3], [4], [4, 5]]
    assert OM.tree_positions(100, par) == [100, 101, 101, 102, 100, 101]
    assert OM.chain_parents(4) == [-1, 0, 1, 2]
    for bad in ([0], [-1, 1], [-1, 5, 0], [-2]):
        with pytest.raises(ValueError):
            OM.tree_depths(bad)


@pytest.mark.parametrize("window", [0, 4, 7])
def test_tree_chain_is_the_causal_chain(window):
    """The chain written as a tree gives attention() bit for bit."""
    rng = np.random.default_rng(10 + window)
    dims = _dims()
    S_, T = 10, 5
    q = F.rb(rng.normal(size=(T, 4, 8)))
    K = F.rb(rng.normal(size=(2, S_ + T, 8)))
    V = F.rb(rng.normal(size=(2, S_ + T, 8)))
    a = OM.attention(dims, q, K, V, [S_ + t for t in range(T)], window)
    b = OM.attention_tree(dims, q, K, V, S_, OM.chain_parents(T), window)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("window", [0, 3, 6])
def test_tree_attention_brute_force(window):
    rng = np.random.default_rng(20 + window)
    dims = _dims()
    S_ = 9
    par = [-1, 0, 0, 1, -1, 4, 3, 6]
    T = len(par)
    q = F.rb(rng.normal(size=(T, 4, 8)))
    K = F.rb(rng.normal(size=(2, S_ + T, 8)))
    V = F.rb(rng.normal(size=(2, S_ + T, 8)))
    got = OM.attention_tree(dims, q, K, V, S_, par, window)
    want = brute_tree_attention(q, K, V, S_, par, window, G=2)
    assert np.all(np.abs(got - want) <= np.abs(want) * 2 ** -8 + 1e-300)


def test_tree_attention_sees_only_ancestors():
    """Changing the K/V rows of a slot that is not an ancestor of t leaves
    t's output bit-identical; changing an ancestor's row changes it."""
    rng = np.random.default_rng(7)
    dims = _dims()
    S_ = 12
    par = [-1, 0, 0, 1, 2, -1]
    T = len(par)
    q = F.rb(rng.normal(size=(T, 4, 8)))
    K = F.rb(rng.normal(size=(2, S_ + T, 8)))
    V = F.rb(rng.normal(size=(2, S_ + T, 8)))
    base = OM.attention_tree(dims, q, K, V, S_, par, 0).reshape(T, -1)
    anc = OM.tree_ancestors(par)
    for u in range(T):
        K2, V2 = K.copy(), V.copy()
        K2[:, S_ + u] += 3.0
        V2[:, S_ + u] += 3.0
        o = OM.attention_tree(dims, q, K2, V2, S_, par, 0).reshape(T, -1)
        for t in range(T):
            if u in anc[t]:
                assert not np.array_equal(o[t], base[t]), (u, t)
            else:
                assert np.array_equal(o[t], base[t]), (u, t)


def test_tree_star_sees_context_and_itself():
    """All slots children of the context: slot t sees the cached rows and its
    own row only, i.e. what a single token at position S sees."""
    rng = np.random.default_rng(11)
    dims = _dims()
    S_, T = 6, 4
    q = F.rb(rng.normal(size=(T, 4, 8)))
    K = F.rb(rng.normal(size=(2, S_ + T, 8)))
    V = F.rb(rng.normal(size=(2, S_ + T, 8)))
    o = OM.attention_tree(dims, q, K, V, S_, [-1] * T, 0).reshape(T, -1)
    for t in range(T):
        Kt = np.concatenate([K[:, :S_], K[:, S_ + t:S_ + t + 1]], axis=1)
        Vt = np.concatenate([V[:, :S_], V[:, S_ + t:S_ + t + 1]], axis=1)
        one = OM.attention(dims, q[t:t + 1], Kt, Vt, [S_], 0).reshape(-1)
        assert np.array_equal(o[t], one)


def _tiny(tokens, cached, window, layers):
    wl = S.scaled(S.WORKLOADS["tiny"], tokens=tokens, cached=cached, windows=(window,) * layers)
    ws = [oracle_weights(S.layer_weights(wl, l), wl) for l in range(layers)]
    caches = [split_cache(S.kv_cache(wl, l)) for l in range(layers)]
    return wl, oracle_dims(wl), ws, caches, np64(S.hidden_state(wl))


def test_tree_decode_step_chain_equivalence():
    """decode_step with the chain given as parents is the default step."""
    wl, dims, ws, caches, h = _tiny(tokens=3, cached=40, window=16, layers=2)
    ca = [(K.copy(), V.copy()) for K, V in caches]
    cb = [(K.copy(), V.copy()) for K, V in caches]
    hA, _ = OM.decode_step(dims, ws, wl.windows, h, ca, wl.positions)
    hB, _ = OM.decode_step(dims, ws, wl.windows, h, cb, wl.positions, parents=OM.chain_parents(3))
    assert np.array_equal(hA, hB)
    for l in range(2):
        assert np.array_equal(ca[l][0], cb[l][0]) and np.array_equal(ca[l][1], cb[l][1])


def test_tree_decode_step_rows_and_positions():
    """A tree step writes slot t's K/V row at S + t, rotated for position
    S + depth(t); slots on different branches do not see each other."""
    wl, dims, ws, caches, h = _tiny(tokens=4, cached=30, window=0, layers=1)
    par = [-1, 0, -1, 2]
    S_ = wl.positions[0]
    c = [(K.copy(), V.copy()) for K, V in caches]
    hT, outs = OM.decode_step(dims, ws, wl.windows, h, c, wl.positions, parents=par)
    q, kr, vr = OM.qkv_project(dims, ws[0], h, [S_ + d for d in OM.tree_depths(par)])
    for t in range(4):
        assert np.array_equal(c[0][0][:, S_ + t], kr[t]) and np.array_equal(c[0][1][:, S_ + t], vr[t])
    # slots 0, 1 (one branch) do not depend on the inputs of slots 2, 3 (the other)
    h2 = h.copy()
    h2[2:] += 0.5
    c2 = [(K.copy(), V.copy()) for K, V in caches]
    hT2, _ = OM.decode_step(dims, ws, wl.windows, h2, c2, wl.positions, parents=par)
    assert np.array_equal(hT[:2], hT2[:2])
    assert not np.array_equal(hT[2:], hT2[2:])
