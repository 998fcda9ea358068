"""The captured step (msk_step_graph_capture / msk_step_graph_launch): a
replay must equal msk_decode_step / msk_decode_step_tree bit for bit, for
several steps with different cached lengths and trees, over the buffers
given at capture time."""

import pytest
import torch

import msk_synth as S
from oracle import model as OM
from tests._gpu import Setup

pytestmark = pytest.mark.gpu

TREE16 = [-1, 0, 1, 1, 2, 4, -1, 6, 3, 8, 5, 10, 0, 12, 9, 11]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_decode_step_persistent_gb300 as M
    M.load_library()  # raises if the extension is missing: no fallback


def _direct(st, h0, kv0, prev, cache_len, parents):
    h, kv = h0.clone(), kv0.clone()
    r = torch.zeros((st.wl.n_layers, st.wl.tokens, st.wl.top_k), dtype=torch.int32, device="cuda")
    if parents is None:
        st.model.decode_step(h, kv, [cache_len + t for t in range(st.wl.tokens)], prev, r)
    else:
        st.model.decode_step_tree(h, kv, cache_len, parents, prev, r)
    return h, kv, r


def test_replay_equals_decode_step():
    wl = S.scaled(S.WORKLOADS["tiny"], tokens=16, cached=300, windows=(8, 0, 8, 8))
    st = Setup(wl, gamma_std=0.1)
    kv0, h0 = st.fresh_kv(), st.hidden()
    prev = torch.zeros((wl.n_layers, wl.tokens, wl.top_k), dtype=torch.int32, device="cuda")
    # the graph's own buffers
    hg, kvg = h0.clone(), kv0.clone()
    rg = torch.zeros_like(prev)
    st.model.capture_step(hg, kvg, prev, rg)
    for cache_len, parents in ((300, None), (250, TREE16), (299, OM.chain_parents(16)), (120, [-1] * 16)):
        hg.copy_(h0)
        kvg.copy_(kv0)
        st.model.replay_step(cache_len, parents)
        h, kv, r = _direct(st, h0, kv0, prev, cache_len, parents)
        assert torch.equal(hg, h), (cache_len, parents)
        assert torch.equal(kvg, kv), (cache_len, parents)
        assert torch.equal(rg, r), (cache_len, parents)
    st.model.close()


def test_replay_full_width_two_layers():
    """The 4096-wide layers (sliding then global) with the routing of the
    previous step fed back, as the bench runs them."""
    wl = S.scaled(S.WORKLOADS["sliding"], windows=(2048, 0))
    st = Setup(wl, gen_device="cuda")
    kv0, h0 = st.fresh_kv(), st.hidden()
    prev = torch.zeros((wl.n_layers, wl.tokens, wl.top_k), dtype=torch.int32, device="cuda")
    _, _, prev_r = _direct(st, h0, kv0, None, wl.cached, None)
    prev.copy_(prev_r)
    hg, kvg = h0.clone(), kv0.clone()
    rg = torch.zeros_like(prev)
    st.model.capture_step(hg, kvg, prev, rg)
    st.model.replay_step(wl.cached, TREE16)
    h, kv, r = _direct(st, h0, kv0, prev, wl.cached, TREE16)
    assert torch.equal(hg, h) and torch.equal(kvg, kv) and torch.equal(rg, r)
    st.model.close()


def test_replay_errors():
    import moe_decode_step_persistent_gb300 as M
    wl = S.scaled(S.WORKLOADS["tiny"], tokens=4, cached=50, windows=(0,))
    st = Setup(wl)
    assert st.model.replay_step(50, check=False) == M.MSK_ERR_NOT_LOADED
    kv, h = st.fresh_kv(), st.hidden()
    st.model.capture_step(h, kv)
    assert st.model.replay_step(wl.max_seq - 3, check=False) == M.MSK_ERR_INVALID_ARG
    assert st.model.replay_step(10, [0, 0, 1, 2], check=False) == M.MSK_ERR_INVALID_ARG
    assert st.model.replay_step(10) == M.MSK_OK
    st.model.close()
