"""Seeded synthetic inputs for the verify step (shared by tests, bench, oracle).

This module draws random tensors with the workloads' shapes and value
distributions.  It holds none of the method's arithmetic: no rounding rule,
quantiser, norm, projection or routing step lives here.  NVFP4 expert weights
are drawn directly as codes (E2M1 nibbles from a fixed categorical law, E4M3
block-scale codes uniform over a fixed code range, and a per-matrix fp32
tensor scale), so neither side's quantiser is involved in making them.

Every tensor is drawn from its own ``torch.Generator`` seeded by
(workload seed, layer, tensor id), so any layer can be regenerated alone, on
the CPU or directly on a CUDA device.  CPU and CUDA generators give different
streams: a test that compares the two paths generates once and copies.

Workloads (the stand-in for the pages' single GSM8K request, which is not
used: batch size one, 16 verify tokens, synthetic weights and activations):
  tiny     1 token, hidden 256, 4 q / 1 kv heads, head_dim 64, global
           attention over 128 cached tokens, pooled 128, 16 experts top-2,
           inter 128.
  sliding  16 tokens, hidden 4096, 32 q / 8 kv heads, head_dim 128, window
           2048 over 4096 cached tokens, pooled 2048, 256 experts top-8,
           inter 1024, Zipf(s=1.1) router bias.
  global   as sliding, global attention over 32768 cached tokens.
  stack8   8 layers (sliding x3, global) x2, 8192 cached tokens.
  full62   62 layers, 46 sliding + 16 global (a global layer after every 3
           sliding ones while globals remain: layers 3, 7, ..., 59 and 61),
           16384 cached tokens.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

# ----------------------------------------------------------------------------
# workload table
# ----------------------------------------------------------------------------


@dataclass(frozen=True)
class Workload:
    name: str
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    pooled: int
    n_experts: int
    top_k: int
    inter: int
    tokens: int
    cached: int
    windows: tuple  # per layer; 0 = global attention
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    zipf_s: float = 1.1  # router bias b_i = -s * ln(rank_i); 0 disables
    weight_std: float = 0.02
    seed: int = 0

    @property
    def n_layers(self) -> int:
        return len(self.windows)

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def max_seq(self) -> int:
        return self.cached + self.tokens

    @property
    def positions(self) -> list:
        return [self.cached + t for t in range(self.tokens)]


def full62_windows(n_layers=62, n_global=16, window=2048):
    """One global layer after every three sliding layers while globals
    remain; the rest sliding.  A literal (SSSG) x 16 needs 64 layers, so the
    16th global is the last layer: globals at 3, 7, ..., 59 and 61."""
    w = [window] * n_layers
    g = [4 * i + 3 for i in range(n_global - 1)] + [n_layers - 1]
    for l in g:
        w[l] = 0
    return tuple(w)


WORKLOADS = {
    "tiny": Workload("tiny", 256, 4, 1, 64, 128, 16, 2, 128, 1, 128, (0,), zipf_s=0.0),
    "sliding": Workload("sliding", 4096, 32, 8, 128, 2048, 256, 8, 1024, 16, 4096, (2048,)),
    "global": Workload("global", 4096, 32, 8, 128, 2048, 256, 8, 1024, 16, 32768, (0,)),
    "stack8": Workload("stack8", 4096, 32, 8, 128, 2048, 256, 8, 1024, 16, 8192,
                       (2048, 2048, 2048, 0, 2048, 2048, 2048, 0)),
    "full62": Workload("full62", 4096, 32, 8, 128, 2048, 256, 8, 1024, 16, 16384,
                       full62_windows()),
}


def scaled(wl: Workload, **kw) -> Workload:
    """A copy of a workload with some fields replaced (small test shapes)."""
    d = dict(wl.__dict__)
    d.update(kw)
    return Workload(**d)


# ----------------------------------------------------------------------------
# generators
# ----------------------------------------------------------------------------

_TENSOR_IDS = {
    "attn_norm": 1, "moe_norm": 2, "w_qkv": 3, "w_o": 4, "w_pool": 5, "w_router": 6,
    "router_bias": 7, "w_unpool": 8, "gate": 9, "up": 10, "down": 11, "hidden": 12,
    "k_cache": 13, "v_cache": 14, "prev_routing": 15,
}


def _gen(seed: int, layer: int, tid: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + (layer + 1) * 7919 + tid * 104_729) & 0x7FFF_FFFF_FFFF)
    return g


def normal_bf16(shape, std, gen, device):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    return (x * std).to(torch.bfloat16)


#: E2M1 magnitude codes 0..7 drawn with these weights (out of 256): the
#: shape of a Gaussian block scaled so its largest element lands near 6.
E2M1_CODE_WEIGHTS = (18, 33, 33, 31, 44, 46, 36, 15)
#: E4M3 block-scale codes drawn uniformly from this inclusive code range
#: (values 96 .. 240).
E4M3_SCALE_CODE_RANGE = (0x6C, 0x77)
#: per-matrix tensor scale: this base value times U(0.8, 1.25); with the two
#: laws above the dequantised weights have a standard deviation near 0.02.
TENSOR_SCALE_BASE = 4.4e-5


def _nibble_lut(device):
    mags = []
    for code, w in enumerate(E2M1_CODE_WEIGHTS):
        mags += [code] * w
    lut = torch.tensor(mags + [m | 8 for m in mags], dtype=torch.uint8, device=device)
    return lut  # index: (sign bit << 8) | byte


def nvfp4_batch(n, rows, cols, gen, device, chunk=8):
    """n NVFP4 matrices [rows][cols]: returns (packed uint8 [n][rows][cols/2],
    scales uint8 [n][rows][cols/16], tensor_scale float32 [n])."""
    lut = _nibble_lut(device)
    packed = torch.empty((n, rows, cols // 2), dtype=torch.uint8, device=device)
    for i0 in range(0, n, chunk):
        i1 = min(n, i0 + chunk)
        idx = torch.randint(0, 512, (i1 - i0, rows, cols), generator=gen, device=device,
                            dtype=torch.int32)
        codes = lut[idx.long()]
        packed[i0:i1] = codes[..., 0::2] | (codes[..., 1::2] << 4)
        del idx, codes
    lo, hi = E4M3_SCALE_CODE_RANGE
    scales = torch.randint(lo, hi + 1, (n, rows, cols // 16), generator=gen, device=device,
                           dtype=torch.int32).to(torch.uint8)
    u = torch.rand((n,), generator=gen, device=device, dtype=torch.float32)
    ts = TENSOR_SCALE_BASE * (0.8 + 0.45 * u)
    return packed, scales, ts.to(torch.float32)


def zipf_bias(n_experts, s, gen, device):
    """Per-expert logit bias -s * ln(r), r a seeded permutation of 1..E, so
    exp(bias) follows a Zipf law of exponent s over a random expert order."""
    if s == 0:
        return torch.zeros(n_experts, dtype=torch.float32, device=device)
    perm = torch.randperm(n_experts, generator=gen, device=device) + 1
    return (-s * torch.log(perm.to(torch.float64))).to(torch.float32)


@dataclass
class LayerTensors:
    """One layer's weights in the caller-facing formats (row-major)."""

    attn_norm: torch.Tensor
    moe_norm: torch.Tensor
    w_qkv: torch.Tensor
    w_o: torch.Tensor
    w_pool: torch.Tensor
    w_router: torch.Tensor
    router_bias: torch.Tensor
    w_unpool: torch.Tensor
    gate: tuple  # (packed [E][I][P/2], scales [E][I][P/16], ts [E])
    up: tuple
    down: tuple  # (packed [E][P][I/2], scales [E][P][I/16], ts [E])
    extra: dict = field(default_factory=dict)


def layer_weights(wl: Workload, layer: int, device="cpu", gamma_std=0.0) -> LayerTensors:
    """Seeded weights of one layer.  Dense N(0, std) bf16; norm weights 1
    (or 1 + N(0, gamma_std) when a test asks for non-trivial gains)."""
    D, P, E, I = wl.hidden, wl.pooled, wl.n_experts, wl.inter
    sd, s = wl.weight_std, wl.seed

    def g(name):
        return _gen(s, layer, _TENSOR_IDS[name], device)

    def gamma(name):
        if gamma_std == 0:
            return torch.ones(D, dtype=torch.bfloat16, device=device)
        return (1.0 + gamma_std * torch.randn(D, generator=g(name), device=device)).to(torch.bfloat16)

    return LayerTensors(
        attn_norm=gamma("attn_norm"),
        moe_norm=gamma("moe_norm"),
        w_qkv=normal_bf16((wl.qkv_rows, D), sd, g("w_qkv"), device),
        w_o=normal_bf16((D, wl.n_q_heads * wl.head_dim), sd, g("w_o"), device),
        w_pool=normal_bf16((P, D), sd, g("w_pool"), device),
        w_router=normal_bf16((E, P), sd, g("w_router"), device),
        router_bias=zipf_bias(E, wl.zipf_s, g("router_bias"), device),
        w_unpool=normal_bf16((D, P), sd, g("w_unpool"), device),
        gate=nvfp4_batch(E, I, P, g("gate"), device),
        up=nvfp4_batch(E, I, P, g("up"), device),
        down=nvfp4_batch(E, P, I, g("down"), device),
    )


def hidden_state(wl: Workload, step: int = 0, device="cpu") -> torch.Tensor:
    """Layer-0 input h [T][D], N(0, 1) bf16, seeded by the step."""
    return normal_bf16((wl.tokens, wl.hidden), 1.0, _gen(wl.seed + 7 * step, -1, _TENSOR_IDS["hidden"], device), device)


def kv_cache(wl: Workload, layer: int, device="cpu") -> torch.Tensor:
    """One layer's cache [2][Hkv][max_seq][d] bf16; the first ``cached``
    positions N(0, 1), the verify positions zero (the step writes them)."""
    shape = (2, wl.n_kv_heads, wl.max_seq, wl.head_dim)
    kv = torch.zeros(shape, dtype=torch.bfloat16, device=device)
    gk = _gen(wl.seed, layer, _TENSOR_IDS["k_cache"], device)
    kv[:, :, : wl.cached] = normal_bf16((2, wl.n_kv_heads, wl.cached, wl.head_dim), 1.0, gk, device)
    return kv


def fill_kv_cache(wl: Workload, layer: int, out: torch.Tensor):
    """As :func:`kv_cache`, written into ``out`` ([2][Hkv][max_seq][d] view
    of a larger cache) on its device."""
    gk = _gen(wl.seed, layer, _TENSOR_IDS["k_cache"], out.device)
    out[:, :, : wl.cached] = normal_bf16((2, wl.n_kv_heads, wl.cached, wl.head_dim), 1.0, gk, out.device)
    out[:, :, wl.cached:] = 0


def random_routing(wl: Workload, seed: int, device="cpu") -> torch.Tensor:
    """A plausible previous-step routing [L][T][k] int32 (distinct experts per
    token), for prefetch tests."""
    g = _gen(wl.seed + seed, -2, _TENSOR_IDS["prev_routing"], device)
    out = torch.empty((wl.n_layers, wl.tokens, wl.top_k), dtype=torch.int32, device=device)
    for l in range(wl.n_layers):
        for t in range(wl.tokens):
            out[l, t] = torch.randperm(wl.n_experts, generator=g, device=device)[: wl.top_k].to(torch.int32)
    return out


def describe(wl: Workload) -> dict:
    return {k: (list(v) if isinstance(v, tuple) else v) for k, v in wl.__dict__.items()}


__all__ = ["Workload", "WORKLOADS", "scaled", "layer_weights", "hidden_state", "kv_cache",
           "fill_kv_cache", "random_routing", "nvfp4_batch", "zipf_bias", "full62_windows",
           "describe", "LayerTensors"]
