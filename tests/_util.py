"""Test helpers: turn generator tensors into oracle inputs, compare tensors."""

from __future__ import annotations

import numpy as np
import torch

from oracle import model as OM


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float32).numpy().astype(np.float64)


def oracle_dims(wl) -> OM.Dims:
    return OM.Dims(hidden=wl.hidden, n_q_heads=wl.n_q_heads, n_kv_heads=wl.n_kv_heads,
                   head_dim=wl.head_dim, pooled=wl.pooled, n_experts=wl.n_experts,
                   top_k=wl.top_k, inter=wl.inter, rms_eps=wl.rms_eps, rope_theta=wl.rope_theta)


def _experts(trip, cols):
    packed, scales, ts = (x.detach().cpu() for x in trip)
    return [OM.Expert(packed[e].numpy(), scales[e].numpy(), float(ts[e]), cols)
            for e in range(packed.shape[0])]


def oracle_weights(lt, wl) -> OM.LayerWeights:
    return OM.LayerWeights(
        attn_norm=np64(lt.attn_norm), moe_norm=np64(lt.moe_norm), w_qkv=np64(lt.w_qkv),
        w_o=np64(lt.w_o), w_pool=np64(lt.w_pool), w_router=np64(lt.w_router),
        router_bias=lt.router_bias.detach().cpu().numpy().astype(np.float64),
        w_unpool=np64(lt.w_unpool),
        gate=_experts(lt.gate, wl.pooled), up=_experts(lt.up, wl.pooled),
        down=_experts(lt.down, wl.inter))


def split_cache(kv: torch.Tensor):
    """[2][Hkv][S][d] bf16 -> (K, V) float64 numpy (copies)."""
    a = np64(kv)
    return a[0].copy(), a[1].copy()


def rel_stats(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) or 1.0
    maxabs = float(np.max(np.abs(got - ref))) if got.size else 0.0
    cos = float(np.dot(got.ravel(), ref.ravel()) /
                (np.linalg.norm(got.ravel()) * np.linalg.norm(ref.ravel()) + 1e-300))
    return maxabs / rms, cos


def within_one_bf16_ulp(got, ref, abs_floor_rel=1e-3, steps=1):
    """True if every element of a bf16 result is within `steps` bf16 rounding
    steps of the float64 reference (2^-7 relative to the element's binade),
    plus an absolute floor of abs_floor_rel * RMS(ref) for elements near zero
    (where fp32 accumulation noise exceeds one ulp of a tiny value)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    _, e = np.frexp(np.maximum(np.abs(ref), 1e-30))
    ulp = np.ldexp(1.0, e - 8)
    floor = abs_floor_rel * float(np.sqrt(np.mean(ref * ref)))
    return bool(np.all(np.abs(got - ref) <= steps * ulp + floor))


def assert_close(got, ref, name, tol_rel=2e-2, min_cos=0.999, ulp_ok=False, ulp_steps=1):
    """The acceptance bar on bf16 outputs: max|err| <= 2e-2 * RMS(ref) and
    cosine >= 0.999.  With ulp_ok, a result whose every element is within one
    bf16 rounding step of the reference also passes (cosine still required):
    a tensor with a high crest factor exceeds 2e-2 * RMS from a single
    rounding step at its largest element."""
    r, c = rel_stats(got, ref)
    ok = r <= tol_rel and c >= min_cos
    if not ok and ulp_ok:
        ok = c >= min_cos and within_one_bf16_ulp(got, ref, steps=ulp_steps)
    assert ok, f"{name}: max|err|/rms={r:.3e} cos={c:.6f}"
    return r, c
