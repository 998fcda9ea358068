"""Per-phase timeline of the layer kernel inside decode steps.

An 8-layer step with the full-size layer's dimensions (16 verify tokens,
16,384 cached tokens, windows S S S G S S S G, routing carried from step to
step).  After six untimed steps (the first also reports the CUDA-event time
of every launch), two steps run in the timing build: every block stamps
%globaltimer at each phase boundary.  For three launches (a sliding layer
followed by a sliding one, a sliding layer followed by a global one, a
global layer) it prints, per stamp, the median / min / max over the blocks
in microseconds after the launch's first block started.  The timing build is
for breakdowns only; its launches run a little slower than untimed ones, and
the script reports by how much: the median step time with and without the
stamps, (with - without) / without, and the difference per launch.

  python -m moe_decode_step_persistent_gb300.micro.timeline
"""

from __future__ import annotations

import sys

import torch

TIMELINE_SLOTS = 64
_PHASES = ["start", "pro_qkv", "attn", "combine", "oproj", "pool", "router", "topk", "gemm1", "gemm2", "mcomb",
           "unpool", "qkv", "end"]
_DENSE = ["qkvcur", "oproj", "pool", "router", "unpool", "qkvnxt"]


def slot_names() -> dict:
    """Stamp slots of the layer kernel: phase starts, 16 + phase for a
    block's work in a phase done, 32 + 4 k + {entry, first tile, end} for the
    k-th dense projection, 56.. for the expert GEMMs, and single stamps."""
    names = {i: p for i, p in enumerate(_PHASES)}
    names.update({16 + i: f"done_{p}" for i, p in enumerate(_PHASES)})
    for k, n in enumerate(_DENSE):
        for j, s in enumerate(["entry", "tile0", "end"]):
            names[32 + 4 * k + j] = f"d_{n}_{s}"
    for j, s in ((0, "g1_staged"), (2, "g1_done"), (3, "g2_staged"), (5, "g2_done")):
        names[56 + j] = s
    names.update({14: "topk_chosen", 15: "dispatch_ready", 30: "w0_logits", 31: "w0_topk",
                  29: "k_entry", 16: "k_dep_done", 47: "rms_stats", 51: "rms_scaled", 35: "attn_kv1", 39: "attn_merge_smem", 43: "attn_partial_out", 55: "attn_q", 62: "attn_kv0", 63: "attn_keys_done"})
    return names


def report(t, title, names):
    t = t.double()
    t0 = t[:, 0][t[:, 0] > 0].min()
    print(f"=== {title}  end max {((t[:, 13] - t0).max() / 1e3):.1f} us")
    rows = []
    for s in range(t.shape[1]):
        v = t[:, s][t[:, s] > 0]
        if v.numel() == 0:
            continue
        v = (v - t0) / 1e3
        rows.append((float(v.median()), s, float(v.min()), float(v.max())))
    for med, s, mn, mx in sorted(rows):
        print(f"  {names.get(s, s):>18} [{s:2d}]  med {med:7.1f}  min {mn:7.1f}  max {mx:7.1f}")


def main(argv=None) -> int:
    import argparse
    import msk_synth as S
    from moe_decode_step_persistent_gb300 import Model

    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--prefetch-experts", type=int, default=14, help="hot experts prefetched into L2 per layer")
    args = ap.parse_args(argv)
    wl = S.scaled(S.WORKLOADS["full62"], windows=(2048, 2048, 2048, 0, 2048, 2048, 2048, 0))
    m = Model(wl, prefetch_experts=args.prefetch_experts)
    for l in range(wl.n_layers):
        lt = S.layer_weights(wl, l, device="cuda")
        m.load_layer(l, lt)
        del lt
    torch.cuda.empty_cache()
    kv = torch.empty((wl.n_layers, 2, wl.n_kv_heads, wl.max_seq, wl.head_dim), dtype=torch.bfloat16, device="cuda")
    for l in range(wl.n_layers):
        S.fill_kv_cache(wl, l, kv[l])
    L, T, k = wl.n_layers, wl.tokens, wl.top_k
    rout = [torch.zeros((L, T, k), dtype=torch.int32, device="cuda") for _ in range(2)]
    hs = [S.hidden_state(wl, step=s, device="cuda") for s in range(8)]
    m.set_launch_timing(True)
    for s in range(6):
        m.decode_step(hs[s].clone(), kv, wl.positions, rout[(s + 1) % 2] if s else None, rout[s % 2])
    print("CUDA-event us per launch (last untimed step):", [round(x * 1e3, 1) for x in m.launch_ms()])
    m.set_launch_timing(False)

    def step_ms(timing, n=6):
        """Median CUDA-event time of n steps with the timing build on / off."""
        m.set_timing(timing)
        ts = []
        for s in range(n):
            h = hs[s % len(hs)].clone()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            m.decode_step(h, kv, wl.positions, rout[(s + 1) % 2], rout[s % 2])
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return sorted(ts)[n // 2]

    off1, on, off2 = step_ms(False), step_ms(True), step_ms(False)
    off = (off1 + off2) / 2
    print(f"instrumentation: step {off:.3f} ms without stamps, {on:.3f} ms with "
          f"({(on - off) / off * 100:.2f} %, {(on - off) / L * 1e3:.2f} us per launch)")
    m.set_timing(True)
    for s in range(6, 8):
        m.decode_step(hs[s].clone(), kv, wl.positions, rout[(s + 1) % 2], rout[s % 2])
        torch.cuda.synchronize()
    tl = m.timeline().clone()
    names = slot_names()
    # gap between launches: a launch's first block start after the previous
    # launch's last block end
    starts = [float(tl[l][:, 0][tl[l][:, 0] > 0].min()) for l in range(L)]
    ends = [float(tl[l][:, 13].max()) for l in range(L)]
    print("launch gaps (us):", [round((starts[l + 1] - ends[l]) / 1e3, 2) for l in range(L - 1)],
          " launch spans (us):", [round((ends[l] - starts[l]) / 1e3, 1) for l in range(L)])
    # the gap's parts: a launch's blocks entering (set-up done, before the
    # wait on the previous launch) and leaving that wait, after the previous
    # launch's last block end (first / last block of the launch)
    for s, what in ((29, "entry"), (16, "dependency wait done")):
        parts = []
        for l in range(1, L):
            v = tl[l][:, s][tl[l][:, s] > 0].double()
            if v.numel():
                parts.append((round((float(v.min()) - ends[l - 1]) / 1e3, 2), round((float(v.max()) - ends[l - 1]) / 1e3, 2)))
        print(f"  {what} after the previous launch's end (first, last block, us):", parts)
    for l, title in ((0, "layer 0 sliding (prologue; next sliding)"), (1, "layer 1 sliding (next sliding)"),
                     (2, "layer 2 sliding (next global)"),
                     (3, "layer 3 global (next sliding)")):
        report(tl[l], title, names)
    m.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
