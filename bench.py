#!/usr/bin/env python
"""Benchmark of the 16-token speculative-verify decode step (batch size one).

Default workload: the full 62-layer step (46 sliding-window layers with
window 2048 + 16 global layers, 16 verify tokens, 16384 cached tokens,
hidden 4096, 32 q / 8 kv heads, head_dim 128, pooled 2048, 256 NVFP4
experts top-8, inter 1024) on one GPU, 62 persistent launches per step,
routing carried from step to step.  Synthetic seeded weights and inputs
(the pages measure one GSM8K request; the synthetic inputs stand in for it).

Prints ONE JSON line (rank 0).  `value` = verified tokens/s over the timed
steps with inputs resident in HBM, the step replayed as one CUDA graph
(msk_step_graph_launch); `e2e` = the same through the C ABI with the step's
hidden state copied from pinned host memory and h2 + routing read back
every step.  `roofline` reports the layer kernel's algorithmic bytes per
launch over its CUDA-event launch duration (the same steps through
msk_decode_step, one event pair per launch) against the measured HBM copy
bandwidth.  `cpu_baseline` times the float64 CPU oracle on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
N > 1 runs N independent replicas (the path does not shard): launched by
torchrun, one process per GPU, max time over ranks, tokens summed.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "16-token verify step µs & tokens/s at bs1; achieved HBM GB/s vs 8 TB/s"
UNIT = "tokens/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "layer_kernel_traffic.json")
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="full62")
    p.add_argument("--prefetch-experts", type=int, default=14)
    p.add_argument("--router-bias-scale", type=float, default=1.0,
                   help="scale the Zipf router-bias exponent (0.77 spreads the routing to ~49 used experts per layer)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--ncu-case", action="store_true",
                   help="run the small profiling case instead (see ncu_case) and exit")
    return p.parse_args(argv)


# ----------------------------------------------------------------------------
# ranks (independent replicas)
# ----------------------------------------------------------------------------


class Ranks:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.dist = None
        self.dev = "cpu"
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = os.environ.get("MSK_BENCH_BACKEND", "nccl" if torch.cuda.is_available() else "gloo")
            if backend == "nccl":
                torch.cuda.set_device(self.local)
                self.dev = "cuda"
            dist.init_process_group(backend=backend)
            self.dist = dist

    def barrier(self):
        if self.dist is not None:
            if self.dev == "cuda":
                self.dist.barrier(device_ids=[self.local])
            else:
                self.dist.barrier()

    def max(self, x: float) -> float:
        if self.dist is None:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=self.dev)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()


def aggregate(slowest_seconds, tokens_per_rank, world):
    """Whole-job throughput: all ranks' tokens over the slowest rank's time."""
    return tokens_per_rank * world / slowest_seconds


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = sorted(v for v in (num(r[1]) for r in rows) if v is not None)
        mx = [v for v in (num(r[2]) for r in rows) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------
# algorithmic bytes
# ----------------------------------------------------------------------------


def launch_bytes(wl, layer, n_used, prologue):
    """Bytes one launch must move at least: each dense weight once, the used
    experts' NVFP4 codes + block scales once, the visible KV rows once, the KV
    and query writes, and the activations in and out."""
    D, P, E, I, T, hd = wl.hidden, wl.pooled, wl.n_experts, wl.inter, wl.tokens, wl.head_dim
    Hq, Hkv = wl.n_q_heads, wl.n_kv_heads
    qkv = wl.qkv_rows * D * 2
    dense = (D * Hq * hd + P * D + E * P + D * P) * 2
    has_next = layer + 1 < wl.n_layers
    dense += qkv * (int(has_next) + int(prologue))
    expert = n_used * (3 * I * P // 2 + 3 * I * P // 16)
    S0 = wl.cached
    w = wl.windows[layer]
    lo = max(0, S0 - w + 1) if w > 0 else 0
    kv_read = (S0 + T - lo) * Hkv * 2 * hd * 2
    kv_write = T * Hkv * 2 * hd * 2 * (int(has_next) + int(prologue))
    act = 2 * T * D * 2 + (T * Hq * hd * 2 if has_next else 0) + E * 4
    return dense + expert + kv_read + kv_write + act


def source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_decode_step_persistent_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_hbm_peak():
    try:
        with open(PEAKS_FILE) as f:
            v = json.load(f).get("hbm_gbs")
        if v:
            return float(v), "measured"
    except Exception:
        pass
    return FALLBACK_HBM_GBS, "fallback"


def traffic_per_launch(workload):
    """DRAM bytes per launch from an ncu capture, if the capture was taken of
    the current kernel sources (else null)."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        if t.get("source_hash") == source_hash() and t.get("workload") == workload:
            return t.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


# ----------------------------------------------------------------------------
# CPU oracle sample
# ----------------------------------------------------------------------------


CPU_SAMPLE_LAYERS = [0, 1, 2, 3, 4, 7]


def oracle_sample(wl, layers):
    """Times one oracle launch per layer in `layers` (float64 numpy on the
    host cores) and returns {layer: seconds}.  Weights are drawn on the GPU
    when one is present (faster) and copied to the host."""
    import torch
    import msk_synth as S
    from oracle import model as OM
    from tests._util import np64, oracle_dims, oracle_weights

    dims = oracle_dims(wl)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    out = {}
    for l in layers:
        lt = S.layer_weights(wl, l, device=dev)
        cpu = S.LayerTensors(
            attn_norm=lt.attn_norm.cpu(), moe_norm=lt.moe_norm.cpu(), w_qkv=lt.w_qkv.cpu(), w_o=lt.w_o.cpu(),
            w_pool=lt.w_pool.cpu(), w_router=lt.w_router.cpu(), router_bias=lt.router_bias.cpu(),
            w_unpool=lt.w_unpool.cpu(), gate=tuple(x.cpu() for x in lt.gate), up=tuple(x.cpu() for x in lt.up),
            down=tuple(x.cpu() for x in lt.down))
        del lt
        w = oracle_weights(cpu, wl)
        kv = S.kv_cache(wl, l, device=dev).cpu()
        K, V = np64(kv[0]), np64(kv[1])
        h = np64(S.hidden_state(wl, device="cpu"))
        q, kr, vr = OM.qkv_project(dims, w, h, wl.positions)
        OM.write_kv(K, V, kr, vr, wl.positions)
        t0 = time.perf_counter()
        OM.launch(dims, w, w, q, h, K, V, wl.positions, wl.windows[l])
        out[l] = time.perf_counter() - t0
        del w, K, V, cpu
    return out


def oracle_step_estimate(wl, times):
    """Step seconds estimated from sampled launch times by layer kind."""
    sl = [t for l, t in times.items() if wl.windows[l] > 0]
    gl = [t for l, t in times.items() if wl.windows[l] == 0]
    ts = sum(sl) / len(sl) if sl else sum(gl) / len(gl)
    tg = sum(gl) / len(gl) if gl else ts
    n_s = sum(1 for w in wl.windows if w > 0)
    return n_s * ts + (wl.n_layers - n_s) * tg


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def blas_threads():
    """Threads numpy's BLAS runs with (threadpoolctl when present, else the
    usual environment variables, else all host cores: the BLAS default)."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v)
    return cpu_threads()


def workload_config(wl, world):
    """The `config` object both arms print: the workload and its dimensions."""
    return {"workload": wl.name, "layers": wl.n_layers, "sliding_layers": sum(1 for w in wl.windows if w > 0),
            "window": max(wl.windows), "verify_tokens": wl.tokens, "cached_tokens": wl.cached,
            "hidden": wl.hidden, "q_heads": wl.n_q_heads, "kv_heads": wl.n_kv_heads,
            "head_dim": wl.head_dim, "pooled": wl.pooled, "experts": wl.n_experts, "top_k": wl.top_k,
            "inter": wl.inter, "zipf_s": wl.zipf_s, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (each step streams ~19 GB)"}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------


def run_ours(args, rk: Ranks):
    import torch
    import msk_synth as S
    from moe_decode_step_persistent_gb300 import Model

    dev = rk.local
    torch.cuda.set_device(dev)
    wl = S.WORKLOADS[args.workload]
    if args.router_bias_scale != 1.0:
        wl = S.scaled(wl, zipf_s=wl.zipf_s * args.router_bias_scale)
    model = Model(wl, prefetch_experts=args.prefetch_experts)
    for l in range(wl.n_layers):
        lt = S.layer_weights(wl, l, device="cuda")
        model.load_layer(l, lt)
        del lt
    torch.cuda.empty_cache()
    kv = torch.empty((wl.n_layers, 2, wl.n_kv_heads, wl.max_seq, wl.head_dim), dtype=torch.bfloat16,
                     device="cuda")
    for l in range(wl.n_layers):
        S.fill_kv_cache(wl, l, kv[l])
    L, T, k = wl.n_layers, wl.tokens, wl.top_k
    nsteps = args.warmup + args.steps
    hid = [S.hidden_state(wl, step=s, device="cuda") for s in range(nsteps)]
    rout = [torch.zeros((L, T, k), dtype=torch.int32, device="cuda") for _ in range(nsteps)]
    pos = wl.positions
    torch.cuda.synchronize()

    for s in range(args.warmup):
        model.decode_step(hid[s], kv, pos, rout[s - 1] if s > 0 else None, rout[s])
    torch.cuda.synchronize()

    # (1) per-launch durations for the roofline: the same steps through
    # msk_decode_step with a CUDA event pair around every launch
    model.set_launch_timing(True)
    launch_ms = []
    for s in range(args.warmup, nsteps):
        model.decode_step(hid[s], kv, pos, rout[s - 1], rout[s])
        launch_ms += model.launch_ms()
    torch.cuda.synchronize()
    model.set_launch_timing(False)
    used, launch_b = [], []
    for s in range(args.warmup, nsteps):
        r = rout[s].cpu()
        for l in range(L):
            u = int(torch.unique(r[l]).numel())
            used.append(u)
            launch_b.append(launch_bytes(wl, l, u, l == 0))

    # (2) the headline: the step captured once as a CUDA graph over fixed
    # buffers and replayed per step (msk_step_graph_launch); each step's
    # hidden state is copied into the graph's input buffer and its routing
    # is carried to the next step inside the timed region
    h_g = torch.empty_like(hid[0])
    prev_g = rout[args.warmup - 1].clone() if args.warmup > 0 else torch.zeros_like(rout[0])
    out_g = torch.zeros_like(rout[0])
    model.capture_step(h_g, kv, prev_g, out_g)

    def graph_step(s):
        h_g.copy_(hid[s])
        model.replay_step(wl.cached)
        prev_g.copy_(out_g)

    for s in range(args.warmup):
        graph_step(s)
    clocks = ClockSampler(dev)
    clocks.start()
    time.sleep(0.3)
    rk.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for s in range(args.warmup, nsteps):
        graph_step(s)
    ev1.record()
    torch.cuda.synchronize()
    rk.barrier()
    clk = clocks.stop()
    elapsed = rk.max(ev0.elapsed_time(ev1) / 1e3)

    # end to end through host buffers: hidden state in from pinned host
    # memory, h2 and the routing back, every step, through the same graph
    e2e = None
    if not args.no_e2e:
        h_host = [hid[s].cpu().pin_memory() for s in range(nsteps)]
        h2_host = torch.empty((T, wl.hidden), dtype=torch.bfloat16).pin_memory()
        r_host = torch.empty((L, T, k), dtype=torch.int32).pin_memory()

        def e2e_step(s):
            h_g.copy_(h_host[s], non_blocking=True)
            model.replay_step(wl.cached)
            h2_host.copy_(h_g, non_blocking=True)
            r_host.copy_(out_g, non_blocking=True)
            prev_g.copy_(out_g)
            torch.cuda.current_stream().synchronize()

        for s in range(args.warmup):
            e2e_step(s)
        rk.barrier()
        t0 = time.perf_counter()
        for s in range(args.warmup, nsteps):
            e2e_step(s)
        t_e2e = rk.max(time.perf_counter() - t0)
        e2e = {"value": aggregate(t_e2e, T * args.steps, rk.world), "unit": UNIT,
               "h2d_bytes_per_step": int(h_host[0].numel() * 2),
               "d2h_bytes_per_step": int(h2_host.numel() * 2 + r_host.numel() * 4)}

    peak, peak_kind = measured_hbm_peak()
    achieved = sum(launch_b) / (sum(launch_ms) / 1e3) / 1e9
    result = {
        "metric": METRIC, "value": aggregate(elapsed, T * args.steps, rk.world), "unit": UNIT,
        "n_gpus": rk.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed / args.steps * 1e3, "us_per_layer": elapsed / args.steps / L * 1e6,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16+nvfp4 (fp32 accumulate)", "data": "synthetic (seeded weights and activations)",
        "config": workload_config(wl, rk.world),
        "run": {"path": "whole step as one CUDA graph (msk_step_graph_launch); roofline launch times from "
                        "the same steps through msk_decode_step with per-launch CUDA events",
                "unique_experts_per_layer_mean": sum(used) / len(used),
                "prefetch_experts": args.prefetch_experts, "router_bias_scale": args.router_bias_scale},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} HBM copy bandwidth",
                     # (captured with the default router bias)
                     "traffic": traffic_per_launch(wl.name) if args.router_bias_scale == 1.0 else None,
                     "bytes_per_launch_mean": sum(launch_b) / len(launch_b),
                     "launch_us_mean": sum(launch_ms) / len(launch_ms) * 1e3},
        "gpu_launches": L * args.steps,
        "clocks": clk,
        "e2e": e2e,
    }
    if rk.rank == 0 and rk.world == 1 and not args.no_cpu_baseline:
        # about 10 s of CPU on a 16-core host: four sliding and two global layers
        times = oracle_sample(wl, CPU_SAMPLE_LAYERS)
        step_s = oracle_step_estimate(wl, times)
        n_sl = sum(1 for l in times if wl.windows[l] > 0)
        n_s = sum(1 for w in wl.windows if w > 0)
        result["cpu_baseline"] = {
            "value": T / step_s, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": f"one float64 numpy oracle launch (multithreaded BLAS, {blas_threads()} threads) each of "
                      f"layers {sorted(times)} ({n_sl} sliding, {len(times) - n_sl} global) of the same "
                      f"workload, {sum(times.values()):.1f} s of CPU; step extrapolated as "
                      f"{n_s} sliding + {wl.n_layers - n_s} global launch estimates"}
    model.close()
    return result


# ----------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ----------------------------------------------------------------------------


def run_reference(args, rk: Ranks):
    """The oracle timed on the host cores.  One timed "step" of this arm is
    one single-layer oracle launch of the workload (a whole 62-layer oracle
    step takes minutes); layers cycle through sliding and global ones.  The
    line's `value` is tokens/s of a whole step extrapolated from the timed
    launches (sliding and global counts from the workload's layer pattern);
    `steps` and `ms_per_step` are the launches actually timed and their mean
    duration."""
    import msk_synth as S
    if rk.rank != 0:
        return None
    wl = S.WORKLOADS[args.workload]
    if args.router_bias_scale != 1.0:
        wl = S.scaled(wl, zipf_s=wl.zipf_s * args.router_bias_scale)
    budget_s = 200.0
    for _ in range(args.warmup):
        oracle_sample(S.WORKLOADS["tiny"], [0])
    timed = {}
    t_start = time.perf_counter()
    steps_done, secs = 0, 0.0
    for s in range(args.steps):
        l = (s * 3) % wl.n_layers  # cycles through sliding and global layers
        t = oracle_sample(wl, [l])
        timed.setdefault(l, []).append(t[l])
        secs += t[l]
        steps_done += 1
        if time.perf_counter() - t_start > budget_s:
            break
    flat = {l: sum(v) / len(v) for l, v in timed.items()}
    step_s = oracle_step_estimate(wl, flat)
    value = wl.tokens / step_s
    n_s = sum(1 for w in wl.windows if w > 0)
    n_sl = sum(1 for l in flat if wl.windows[l] > 0)
    sample = (f"{steps_done} single-layer float64 numpy oracle launches (multithreaded BLAS, {blas_threads()} "
              f"threads) of layers {sorted(flat)} ({n_sl} sliding, {len(flat) - n_sl} global), {secs:.1f} s; "
              f"whole step extrapolated as {n_s} sliding + {wl.n_layers - n_s} global launches")
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": rk.world, "steps": steps_done,
        "warmup": args.warmup, "ms_per_step": secs / steps_done * 1e3,
        "step_estimate_ms": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (bf16/nvfp4 storage rounding)", "data": "synthetic",
        "impl": "reference",
        "config": workload_config(wl, rk.world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def ncu_case():
    """Small case for ncu captures (a few GB on the device): a 4-layer model
    with the full 62-layer step's dimensions and 16384 cached tokens, layer
    windows (2048, 2048, 0, 2048).  Launch order: layer 0 (with the
    prologue), layer 1, layer 2, then (layer 1, layer 2) three more times, so
    that `-s 3 -c 2` captures one sliding-window launch (layer 1) and one
    global-attention launch (layer 2), each with the next layer's QKV."""
    import torch
    import msk_synth as S
    from moe_decode_step_persistent_gb300 import Model

    wl = S.scaled(S.WORKLOADS["full62"], windows=(2048, 2048, 0, 2048))
    m = Model(wl)
    for l in range(wl.n_layers):
        lt = S.layer_weights(wl, l, device="cuda")
        m.load_layer(l, lt)
        del lt
    torch.cuda.empty_cache()
    kv = torch.empty((wl.n_layers, 2, wl.n_kv_heads, wl.max_seq, wl.head_dim), dtype=torch.bfloat16, device="cuda")
    for l in range(wl.n_layers):
        S.fill_kv_cache(wl, l, kv[l])
    h = S.hidden_state(wl, device="cuda")
    rout = torch.zeros((wl.n_layers, wl.tokens, wl.top_k), dtype=torch.int32, device="cuda")
    prev = rout.clone()
    m.layer_step(0, h.clone(), kv, wl.positions, None, rout[0], run_prologue=True)
    for _ in range(4):
        for l in (1, 2):
            m.layer_step(l, h.clone(), kv, wl.positions, prev[l], rout[l])
        prev.copy_(rout)
    torch.cuda.synchronize()
    print(json.dumps({"ncu_case": "full62 dims, windows (2048, 2048, 0, 2048)",
                      "device_gb": round(torch.cuda.max_memory_allocated() / 1e9, 2)}))


def main(argv=None):
    args = parse_args(argv)
    if args.ncu_case:
        ncu_case()
        return
    rk = Ranks()
    try:
        res = run_reference(args, rk) if args.impl == "reference" else run_ours(args, rk)
        if rk.rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
    finally:
        rk.close()


if __name__ == "__main__":
    main()
