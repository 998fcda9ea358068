"""bench.py's host arithmetic, on the CPU: the algorithmic bytes per launch
(the roofline numerator) against the byte counts spelled out for the
workload's shapes, and the CPU baseline's step estimate."""

import bench
import msk_synth as S

# per-component counts of the full-size layer (hidden 4096, 32 q / 8 kv heads
# of 128, pooled 2048, 256 experts, intermediate 1024, 16 verify tokens)
QKV = 6144 * 4096 * 2          # 50,331,648
DENSE_NO_QKV = (4096 * 4096 + 2048 * 4096 + 4096 * 2048 + 256 * 2048) * 2  # o, pool, unpool, router
EXPERT = 2 * 1_048_576 + 1_048_576 + 393_216  # gate + up + down fp4 codes, then their E4M3 scales
KV_ROW = 8 * 2 * 128 * 2       # one position's K and V rows over the 8 kv heads, bf16
ACT = 2 * 16 * 4096 * 2 + 256 * 4  # hidden in and out, logits
Q_STASH = 16 * 32 * 128 * 2


def test_dense_and_expert_counts():
    assert QKV + DENSE_NO_QKV == 118_489_088
    assert EXPERT == 3_538_944


def test_sliding_launch_bytes():
    wl = S.WORKLOADS["full62"]
    assert wl.windows[0] == 2048 and wl.cached == 16384
    # keys [16384 - 2047, 16399]: 2,063 visible rows; the next layer's QKV,
    # 16 new KV rows and the query stash are written
    want = QKV + DENSE_NO_QKV + 37 * EXPERT + 2063 * KV_ROW + 16 * KV_ROW + ACT + Q_STASH
    assert bench.launch_bytes(wl, 0, 37, False) == want


def test_global_launch_bytes():
    wl = S.WORKLOADS["full62"]
    assert wl.windows[3] == 0
    want = QKV + DENSE_NO_QKV + 49 * EXPERT + 16400 * KV_ROW + 16 * KV_ROW + ACT + Q_STASH
    assert bench.launch_bytes(wl, 3, 49, False) == want


def test_prologue_and_last_layer():
    wl = S.WORKLOADS["full62"]
    base = bench.launch_bytes(wl, 0, 37, False)
    # the prologue adds this layer's QKV weights and its own KV write
    assert bench.launch_bytes(wl, 0, 37, True) == base + QKV + 16 * KV_ROW
    # the last layer has no next QKV, KV write or query stash
    last = wl.n_layers - 1
    assert wl.windows[last] == 0
    want = DENSE_NO_QKV + 37 * EXPERT + 16400 * KV_ROW + ACT
    assert bench.launch_bytes(wl, last, 37, False) == want


def test_cpu_step_estimate_weights_the_layer_kinds():
    wl = S.WORKLOADS["full62"]
    assert sum(1 for w in wl.windows if w > 0) == 46 and wl.n_layers == 62
    times = {0: 1.0, 1: 3.0, 3: 10.0}  # sliding mean 2, global 10
    assert bench.oracle_step_estimate(wl, times) == 46 * 2.0 + 16 * 10.0
    # the default sample holds both kinds of layer
    assert {wl.windows[l] > 0 for l in bench.CPU_SAMPLE_LAYERS} == {True, False}


def test_reference_line_reports_what_it_timed():
    """The reference arm's `steps` are the single-layer oracle launches it
    timed and `ms_per_step` their mean, so steps x ms_per_step is the time
    actually spent; its `config` is the same object the GPU arm prints."""
    import time
    args = bench.parse_args(["--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "0"])
    t0 = time.perf_counter()
    line = bench.run_reference(args, bench.Ranks())
    elapsed = time.perf_counter() - t0
    assert line["impl"] == "reference" and line["steps"] == 3
    assert line["steps"] * line["ms_per_step"] / 1e3 <= elapsed
    assert line["config"] == bench.workload_config(S.WORKLOADS["tiny"], 1)
    assert line["cpu_baseline"]["value"] == line["value"] and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
