"""The allocation-free attention entry point (msk_attention_noalloc).

It serves callers that cannot allocate device memory when they need
attention (memory handed out only by a framework's own pool, or no
allocation allowed while work is being recorded).  Its scratch is a fixed
array inside the library, shared by every call.  This file is collected last
so that a run stopping at the first failure has run every other test; it
also passes alone in a fresh process.

Checked through the C ABI against the existing entry point -- the attention
output msk_layer_step produces for the same queries and KV cache, bit for
bit (both run the same attention code on the same grid) -- and against the
oracle's attention on the same queries, on two calls in a row (the second
reuses the shared scratch left by the first)."""

import pytest
import torch

import msk_synth as S
from oracle import model as OM
from tests._gpu import Setup, assert_close, read_scratch, split_kv
from tests._util import np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_decode_step_persistent_gb300 as mod
    mod.load_library()
    return mod


@pytest.mark.parametrize("windows", [(2048, 2048), (0, 0)])
def test_noalloc_matches_layer_step(M, windows):
    wl = S.scaled(S.WORKLOADS["tiny"], tokens=16, n_q_heads=8, n_kv_heads=2, head_dim=128, cached=3000,
                  windows=windows)
    st = Setup(wl)
    kv = st.fresh_kv()
    h = st.hidden()
    st.model.layer_step(0, h, kv, wl.positions, run_prologue=True)
    q1 = read_scratch(st, "q")          # layer 1's queries, written by launch 0
    st.model.layer_step(1, h, kv, wl.positions)
    ref = read_scratch(st, "attn_o")    # the existing entry point's attention output
    torch.cuda.synchronize()
    K, V = split_kv(kv[1])
    o_ref = OM.attention(st.dims, np64(q1), K, V, wl.positions, wl.windows[1])
    for _ in range(2):                  # two calls in a row share the scratch
        out = torch.full_like(ref, float("nan"))
        status = M.msk_attention_noalloc(q1, kv[1], wl.cached, wl.windows[1], out)
        assert status == M.MSK_OK
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"no-alloc attention differs from msk_layer_step's, windows {windows}"
        assert_close(np64(out), o_ref, f"no-alloc attention against the oracle, windows {windows}")
    st.model.close()


def test_noalloc_rejects_unsupported_sizes(M):
    q = torch.zeros((17, 8, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((2, 2, 64, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((17, 8 * 128), dtype=torch.bfloat16, device="cuda")
    assert M.msk_attention_noalloc(q, kv, 0, 0, out) == 2  # 17 tokens: beyond the maximum
    q96 = torch.zeros((4, 8, 96), dtype=torch.bfloat16, device="cuda")
    kv96 = torch.zeros((2, 2, 64, 96), dtype=torch.bfloat16, device="cuda")
    out96 = torch.zeros((4, 8 * 96), dtype=torch.bfloat16, device="cuda")
    assert M.msk_attention_noalloc(q96, kv96, 0, 0, out96) == 2  # head_dim 96 unsupported
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    # more kv heads than SMs (each kv head needs a block of its own); also
    # wider than 4096 query columns.  Rejected on the host, before any launch.
    h = nsm + 8
    qh = torch.zeros((1, h, 64), dtype=torch.bfloat16, device="cuda")
    kvh = torch.zeros((2, h, 16, 64), dtype=torch.bfloat16, device="cuda")
    outh = torch.zeros((1, h * 64), dtype=torch.bfloat16, device="cuda")
    assert M.msk_attention_noalloc(qh, kvh, 0, 0, outh) == 2
    # 4096 < n_q_heads * head_dim with few kv heads
    qw = torch.zeros((1, 64, 128), dtype=torch.bfloat16, device="cuda")
    kvw = torch.zeros((2, 1, 16, 128), dtype=torch.bfloat16, device="cuda")
    outw = torch.zeros((1, 64 * 128), dtype=torch.bfloat16, device="cuda")
    assert M.msk_attention_noalloc(qw, kvw, 0, 0, outw) == 2
