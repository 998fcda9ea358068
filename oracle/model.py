"""The verify step as plain float64 numpy: one decoder layer, and the stack.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

What one persistent launch computes ([orcarouter] §Dove si colloca il confine
del kernel; [newruntime] §What happened; [ai4snews] §Interpretation): layer
l's attention through its MoE block, then layer l+1's QKV projection and KV
write.  The megakernel is a scheduling technique; its result is that of the
unfused layer, which is what this module writes out:

  1. x  = rb(RMSNorm(h; g_attn));  qkv = rb(x W_qkv^T), columns
     [q (Hq*d) | k (Hkv*d) | v (Hkv*d)], head-major.
  2. RoPE (rotate-half over the whole head) on q and k; K = rb(k'), V = v are
     written at positions p_t; q' = rb(q') is kept for the next launch.
  3. GQA attention: query head h reads kv head h // (Hq/Hkv); token t sees
     keys j in [max(0, p_t - W + 1), p_t] on sliding layers (window W, "the
     previous 2,048 tokens") or [0, p_t] on global layers; causal inside the
     verify block; scores scaled by 1/sqrt(d); softmax; o = rb(sum p_j V_j).
  4. h1 = rb(h + rb(o W_o^T)).
  5. x2 = rb(RMSNorm(h1; g_moe)); pooled = rb(x2 W_pool^T)  (the pooler that
     shrinks each token vector before the experts).
  6. logits = fp32(fp32(pooled W_r^T) + bias); top-k by (logit desc, index
     asc); gate_r = softmax over the k selected logits.
  7. Per selected (t, e): a = Q4(pooled_t); g = a Wg_e^T; u = a Wu_e^T;
     s = silu(g) * u; s_q = Q4(fp32(s)) (the fp4 intermediate);
     y = rb(s_q Wd_e^T) (the bf16 expert output).
  8. m = rb(sum_r gate_r y_r) in rank order; h2 = rb(h1 + rb(m W_unpool^T))
     (the unpooler restores the token vector; residual).
  9. If a next layer exists: steps 1-2 on h2 with its weights.

Readings where the pages are silent (each listed in the design notes):
pre-norm with two RMSNorms per layer and no projection biases; rotate-half
RoPE over the full head with angles p * theta^(-2i/d) in float64; contiguous
GQA groups; the window boundary p - W + 1; a causal chain inside the verify
block by default, or a tree of candidates given by parent slots (positions
S + depth, rows at S + slot, ancestor-only visibility); the router bias added before both the choice and the softmax; ties in
the top-k go to the lower expert index; W4A4 experts with activation tensor
scale 1; the residual stream stored in bf16.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .formats import f32, nvfp4_dequant, q4, rb


@dataclass(frozen=True)
class Dims:
    """Model dimensions of one layer (the workload definitions fix them)."""

    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    pooled: int
    n_experts: int
    top_k: int
    inter: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim


@dataclass
class Expert:
    """One NVFP4 matrix: packed [rows][cols/2], E4M3 scales [rows][cols/16]."""

    packed: np.ndarray
    scales: np.ndarray
    tensor_scale: float
    cols: int

    def dequant(self) -> np.ndarray:
        return nvfp4_dequant(self.packed, self.scales, self.tensor_scale, self.cols)


@dataclass
class LayerWeights:
    """Weights of one decoder layer, as float64 values of their stored types."""

    attn_norm: np.ndarray  # [D]
    moe_norm: np.ndarray  # [D]
    w_qkv: np.ndarray  # [(Hq+2Hkv)d][D]
    w_o: np.ndarray  # [D][Hq d]
    w_pool: np.ndarray  # [P][D]
    w_router: np.ndarray  # [E][P]
    router_bias: np.ndarray  # [E] float32 values
    w_unpool: np.ndarray  # [D][P]
    gate: list = field(default_factory=list)  # [E] of Expert, [I][P]
    up: list = field(default_factory=list)  # [E] of Expert, [I][P]
    down: list = field(default_factory=list)  # [E] of Expert, [P][I]


# ----------------------------------------------------------------------------
# pieces
# ----------------------------------------------------------------------------


def rmsnorm(h, gamma, eps):
    """rb(h / sqrt(mean(h^2) + eps) * gamma) along the last axis."""
    h = np.asarray(h, dtype=np.float64)
    ms = np.mean(h * h, axis=-1, keepdims=True)
    return rb(h / np.sqrt(ms + eps) * gamma)


def rope(v, positions, theta):
    """Rotate-half RoPE over the whole head.  v: [T][H][d]; positions [T].

    Pair (i, i + d/2), i < d/2, is rotated by angle p * theta^(-2i/d):
    (a, b) -> (a cos - b sin, a sin + b cos).  Float64 throughout; the
    caller rounds.
    """
    v = np.asarray(v, dtype=np.float64)
    d = v.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = np.power(float(theta), -2.0 * i / d)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]  # [T][half]
    cos = np.cos(ang)[:, None, :]
    sin = np.sin(ang)[:, None, :]
    a = v[..., :half]
    b = v[..., half:]
    return np.concatenate([a * cos - b * sin, a * sin + b * cos], axis=-1)


def qkv_project(dims: Dims, w: LayerWeights, h, positions):
    """Steps 1-2: returns (q' [T][Hq][d], K rows [T][Hkv][d], V rows
    [T][Hkv][d]), all bf16 values."""
    T = h.shape[0]
    d, Hq, Hkv = dims.head_dim, dims.n_q_heads, dims.n_kv_heads
    x = rmsnorm(h, w.attn_norm, dims.rms_eps)
    qkv = rb(x @ w.w_qkv.T)
    q = qkv[:, : Hq * d].reshape(T, Hq, d)
    k = qkv[:, Hq * d : (Hq + Hkv) * d].reshape(T, Hkv, d)
    v = qkv[:, (Hq + Hkv) * d :].reshape(T, Hkv, d)
    return rb(rope(q, positions, dims.rope_theta)), rb(rope(k, positions, dims.rope_theta)), v


def write_kv(K, V, k_rows, v_rows, positions):
    """Store the new rows: K/V caches are [Hkv][max_seq][d]."""
    for t, p in enumerate(positions):
        K[:, p, :] = k_rows[t]
        V[:, p, :] = v_rows[t]


def visible_range(p, window):
    """Keys token at position p sees: [lo, p] inclusive."""
    lo = max(0, p - window + 1) if window > 0 else 0
    return lo, p


def attention(dims: Dims, q, K, V, positions, window):
    """Step 3.  q: [T][Hq][d]; K, V: [Hkv][max_seq][d]; returns o [T][Hq*d]."""
    T = q.shape[0]
    d, G = dims.head_dim, dims.group
    o = np.zeros((T, dims.n_q_heads, d))
    scale = 1.0 / np.sqrt(d)
    for t, p in enumerate(positions):
        lo, hi = visible_range(p, window)
        for hq in range(dims.n_q_heads):
            kv = hq // G
            s = (K[kv, lo : hi + 1, :] @ q[t, hq]) * scale
            e = np.exp(s - s.max())
            o[t, hq] = (e / e.sum()) @ V[kv, lo : hi + 1, :]
    return rb(o.reshape(T, -1))


def tree_depths(parents):
    """Depth of every verify slot of a candidate tree: parents[t] is the
    slot of t's parent (-1: a child of the last cached token), always an
    earlier slot; depth = number of verify ancestors."""
    depth = []
    for t, p in enumerate(parents):
        p = int(p)
        if p < -1 or p >= t:
            raise ValueError(f"parents[{t}] = {p}: a parent must be -1 or an earlier slot")
        depth.append(0 if p < 0 else depth[p] + 1)
    return depth


def tree_ancestors(parents):
    """For every slot, the sorted list of verify slots it attends to: its
    ancestors and itself."""
    tree_depths(parents)  # validates
    out = []
    for t in range(len(parents)):
        a, u = [], t
        while u >= 0:
            a.append(u)
            u = int(parents[u])
        out.append(sorted(a))
    return out


def tree_positions(cache_len, parents):
    """Positions of the verify slots: the cached length plus the depth
    ([orcarouter] on the draft: a tree of candidates is verified; a slot at
    depth d continues the context at position S + d)."""
    return [cache_len + d for d in tree_depths(parents)]


def chain_parents(T):
    """The linear chain as a tree: slot t's parent is t - 1."""
    return [t - 1 for t in range(T)]


def attention_tree(dims: Dims, q, K, V, cache_len, parents, window):
    """Step 3 with a tree of candidates.  Slot t (position p_t = S + depth)
    sees the cached keys j < S and the verify rows S + u of its ancestors
    and itself (slot order), each only if its position (j, or S + depth(u))
    lies in the window [p_t - W + 1, p_t] on sliding layers; then as
    attention().  The verify rows are stored at S + slot.  For the chain
    this is attention() exactly."""
    T = q.shape[0]
    d, G = dims.head_dim, dims.group
    S = cache_len
    pos = tree_positions(S, parents)
    anc = tree_ancestors(parents)
    o = np.zeros((T, dims.n_q_heads, d))
    scale = 1.0 / np.sqrt(d)
    for t in range(T):
        lo, _ = visible_range(pos[t], window)
        keys = list(range(min(lo, S), S)) + [S + u for u in anc[t] if pos[u] >= lo]
        for hq in range(dims.n_q_heads):
            kv = hq // G
            s = (K[kv, keys, :] @ q[t, hq]) * scale
            e = np.exp(s - s.max())
            o[t, hq] = (e / e.sum()) @ V[kv, keys, :]
    return rb(o.reshape(T, -1))


def router(dims: Dims, w: LayerWeights, pooled, forced_idx=None):
    """Step 6.  Returns (idx [T][k] int, gates [T][k], logits [T][E] fp32
    values).  With ``forced_idx`` the choice is taken as given (used to
    check downstream tolerance on near-tie tokens) and gates follow it."""
    logits = f32(f32(pooled @ w.w_router.T) + f32(w.router_bias)[None, :])
    T, E = logits.shape
    k = dims.top_k
    if forced_idx is None:
        idx = np.zeros((T, k), dtype=np.int64)
        for t in range(T):
            order = np.lexsort((np.arange(E), -logits[t]))  # logit desc, index asc
            idx[t] = order[:k]
    else:
        idx = np.asarray(forced_idx, dtype=np.int64)
    sel = np.take_along_axis(logits, idx, axis=1)
    top = sel.max(axis=1, keepdims=True)
    ex = np.exp(sel - top)
    gates = ex / ex.sum(axis=1, keepdims=True)
    return idx, gates, logits


def silu(x):
    return x / (1.0 + np.exp(-x))


def experts(dims: Dims, w: LayerWeights, pooled, idx, gates):
    """Steps 7-8 (combine only).  Returns (m [T][P], y [T][k][P], s_q values
    [T][k][I])."""
    T, k = idx.shape
    P, I = dims.pooled, dims.inter
    a = q4(pooled)[2]  # [T][P]
    y = np.zeros((T, k, P))
    sq = np.zeros((T, k, I))
    for e in np.unique(idx):
        sel = np.argwhere(idx == e)  # (t, r) pairs
        wg, wu, wd = w.gate[e].dequant(), w.up[e].dequant(), w.down[e].dequant()
        for t, r in sel:
            g = wg @ a[t]
            u = wu @ a[t]
            s = f32(silu(g) * u)
            sq[t, r] = q4(s)[2]
            y[t, r] = rb(wd @ sq[t, r])
    m = np.zeros((T, P))
    for t in range(T):
        acc = np.zeros(P)
        for r in range(k):  # rank order
            acc = acc + gates[t, r] * y[t, r]
        m[t] = rb(acc)
    return m, y, sq


def launch(dims: Dims, w: LayerWeights, w_next, q, h, K, V, positions, window,
           K_next=None, V_next=None, forced_idx=None, parents=None):
    """One launch: attention(l) .. QKV(l+1) + KV write.

    q: [T][Hq][d] rotated queries of layer l (from the previous launch or the
    prologue); K/V: layer l's caches, already holding the new rows.
    With ``parents`` (a candidate tree), positions[0] is the cached length S,
    the RoPE positions are S + depth and the rows are written at S + slot.
    """
    if parents is None:
        o = attention(dims, q, K, V, positions, window)
        rope_pos, rows = positions, positions
    else:
        S = positions[0]
        o = attention_tree(dims, q, K, V, S, parents, window)
        rope_pos, rows = tree_positions(S, parents), [S + t for t in range(len(parents))]
    h1 = rb(h + rb(o @ w.w_o.T))
    x2 = rmsnorm(h1, w.moe_norm, dims.rms_eps)
    pooled = rb(x2 @ w.w_pool.T)
    idx, gates, logits = router(dims, w, pooled, forced_idx)
    m, y, sq = experts(dims, w, pooled, idx, gates)
    h2 = rb(h1 + rb(m @ w.w_unpool.T))
    out = dict(o=o, h1=h1, pooled=pooled, logits=logits, idx=idx, gates=gates,
               y=y, sq=sq, m=m, h2=h2)
    if w_next is not None:
        qn, kn, vn = qkv_project(dims, w_next, h2, rope_pos)
        out.update(q_next=qn, k_next=kn, v_next=vn)
        if K_next is not None:
            write_kv(K_next, V_next, kn, vn, rows)
    return out


def decode_step(dims: Dims, layers, windows, h, caches, positions, forced_idx=None, parents=None):
    """The whole verify step: prologue (layer 0's QKV + KV write), then one
    launch per layer.  caches: list of (K, V) per layer, modified in place.
    With ``parents`` see launch().  Returns (h_final, per-layer outputs)."""
    if parents is None:
        rope_pos, rows = positions, positions
    else:
        rope_pos = tree_positions(positions[0], parents)
        rows = [positions[0] + t for t in range(len(parents))]
    q, kr, vr = qkv_project(dims, layers[0], h, rope_pos)
    write_kv(caches[0][0], caches[0][1], kr, vr, rows)
    outs = []
    L = len(layers)
    for l in range(L):
        nxt = layers[l + 1] if l + 1 < L else None
        Kn, Vn = (caches[l + 1] if l + 1 < L else (None, None))
        fi = None if forced_idx is None else forced_idx[l]
        o = launch(dims, layers[l], nxt, q, h, caches[l][0], caches[l][1], positions,
                   windows[l], Kn, Vn, fi, parents)
        outs.append(o)
        h = o["h2"]
        if nxt is not None:
            q = o["q_next"]
    return h, outs
