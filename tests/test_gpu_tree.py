"""GPU parity of the tree-of-candidates verification ([orcarouter], the
draft section: the verified block is a tree of candidate tokens), through
msk_layer_step_tree / msk_decode_step_tree, against the oracle's tree
attention.  Same acceptance as test_gpu_parity (stage by stage under teacher
forcing); the chain written as a tree must reproduce the chain entry points
bit for bit."""

import numpy as np
import pytest
import torch

import msk_synth as S
from oracle import model as OM
from tests._gpu import Setup, check_launch, run_layers

pytestmark = pytest.mark.gpu

# a 16-slot candidate tree: two roots, branches of different depths (max 7)
TREE16 = [-1, 0, 1, 1, 2, 4, -1, 6, 3, 8, 5, 10, 0, 12, 9, 11]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_decode_step_persistent_gb300 as M
    M.load_library()  # raises if the extension is missing: no fallback


def _check_tree(wl, parents, gen_device="cpu", gamma_std=0.0):
    """Every launch stage by stage; the first launch's attention (queries
    from its own prologue, not capturable) on cosine, the later ones on the
    queries the GPU used."""
    st = Setup(wl, gen_device=gen_device, gamma_std=gamma_std)
    kv = st.fresh_kv()
    h = st.hidden()
    recs = run_layers(st, h, kv, wl.positions, parents=parents)
    torch.cuda.synchronize()
    rep = []
    for r in recs:
        check_launch(st, r, kv, wl.positions, rep, parents=parents, strict_first_attention=False)
    st.model.close()
    return rep


def test_tree_depths_of_the_fixture():
    assert max(OM.tree_depths(TREE16)) == 7 and OM.tree_depths(TREE16)[6] == 0


def test_chain_as_tree_is_bit_identical():
    """parents[t] = t - 1 through the tree entry points gives exactly the
    chain entry points' hidden state, KV rows and routing."""
    wl = S.scaled(S.WORKLOADS["tiny"], tokens=16, cached=300, windows=(8, 0, 8))
    st = Setup(wl, gamma_std=0.1)
    outs = []
    for parents in (None, OM.chain_parents(16)):
        kv = st.fresh_kv()
        h = st.hidden()
        recs = run_layers(st, h, kv, wl.positions, capture=False, parents=parents)
        torch.cuda.synchronize()
        outs.append((h.clone(), kv.clone(), [r["routing"].clone() for r in recs]))
    (ha, kva, ra), (hb, kvb, rb) = outs
    assert torch.equal(ha, hb) and torch.equal(kva, kvb)
    assert all(torch.equal(x, y) for x, y in zip(ra, rb))
    st.model.close()


def test_tree_small_shapes():
    """A window shorter than the tree's depth (ancestors outside the window
    are masked), a global layer, and a star (every slot a child of the
    context)."""
    wl = S.scaled(S.WORKLOADS["tiny"], tokens=16, cached=200, windows=(5, 0))
    _check_tree(wl, TREE16, gamma_std=0.1)
    _check_tree(wl, [-1] * 16)


def test_tree_sliding_and_global_full_width():
    """The 4096-wide layer with 32 query / 8 kv heads: sliding-window (2048
    over 4096 cached), global, sliding, verifying the tree."""
    wl = S.scaled(S.WORKLOADS["sliding"], windows=(2048, 0, 2048))
    rep = _check_tree(wl, TREE16, gen_device="cuda")
    assert len(rep) == 3


def test_decode_step_tree_equals_launch_sequence():
    """msk_decode_step_tree is the prologue plus one tree launch per layer."""
    wl = S.scaled(S.WORKLOADS["tiny"], tokens=16, cached=120, windows=(16, 0, 16))
    st = Setup(wl)
    kva, ha = st.fresh_kv(), st.hidden()
    ra = torch.zeros((wl.n_layers, wl.tokens, wl.top_k), dtype=torch.int32, device="cuda")
    st.model.decode_step_tree(ha, kva, wl.positions[0], TREE16, None, ra)
    kvb, hb = st.fresh_kv(), st.hidden()
    recs = run_layers(st, hb, kvb, wl.positions, capture=False, parents=TREE16)
    torch.cuda.synchronize()
    assert torch.equal(ha, hb) and torch.equal(kva, kvb)
    for l, r in enumerate(recs):
        assert torch.equal(ra[l], r["routing"])
    st.model.close()


def test_tree_rejects_bad_parents():
    import moe_decode_step_persistent_gb300 as M
    wl = S.scaled(S.WORKLOADS["tiny"], tokens=4, cached=50, windows=(0,))
    st = Setup(wl)
    kv, h = st.fresh_kv(), st.hidden()
    for bad in ([0, 0, 1, 2], [-1, 1, 0, 0], [-1, 0, -2, 1]):
        assert st.model.layer_step_tree(0, h, kv, 50, bad, check=False) == M.MSK_ERR_INVALID_ARG
    assert st.model.layer_step_tree(0, h, kv, wl.max_seq - 3, [-1, 0, 1, 2], check=False) == M.MSK_ERR_INVALID_ARG
    st.model.close()
