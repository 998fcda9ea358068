"""The speculative hot-expert prefetch ranks the right experts.

[ai4snews] "Interpretation": the previous step's routing names the 14
experts used most, and their weights are pulled into L2 before the router
has decided.  Reading of the ranking: counts over the layer's previous
[T][k] routing, descending, ties to the lower expert index, only experts
with a count above zero, at most 14.  The kernel's ranked list (block 0's,
read back through msk_debug_scratch) is compared with that ranking computed
here from the counts; the launch's outputs do not depend on it (checked in
tests/test_gpu_invariants.py)."""

import numpy as np
import pytest
import torch

import msk_synth as S
from tests._gpu import Setup

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import moe_decode_step_persistent_gb300 as M
    M.load_library()


def ranking(prev, want=14):
    counts = np.bincount(np.asarray(prev).ravel(), minlength=256)
    order = sorted((e for e in range(len(counts)) if counts[e] > 0), key=lambda e: (-counts[e], e))
    return order[:want]


def read_ranked(st):
    buf = torch.zeros(33, dtype=torch.int32, device="cuda")
    st.model.debug_scratch(9, buf)
    v = buf.cpu().tolist()
    return v[1:1 + v[0]]


@pytest.mark.parametrize("case", ["ties_and_cap", "few_experts", "none"])
def test_hot_expert_ranking(case):
    wl = S.scaled(S.WORKLOADS["tiny"], tokens=16, cached=64, windows=(0,))
    st = Setup(wl)
    kv = st.fresh_kv()
    h = st.hidden()
    if case == "ties_and_cap":
        # 15 experts used (counts 5, 5, 4, 4, 3, 2, then nine 1s): the cap of
        # 14 drops the highest-indexed expert of count 1
        counts = {7: 5, 3: 5, 12: 4, 1: 4, 0: 3, 9: 2, 15: 1, 4: 1, 2: 1, 5: 1, 6: 1, 8: 1, 10: 1, 11: 1, 13: 1}
        flat = [e for e, c in counts.items() for _ in range(c)]
    elif case == "few_experts":
        flat = [6] * 20 + [2] * 12  # only two experts used
    else:
        flat = None
    prev = None
    if flat is not None:
        assert len(flat) == wl.tokens * wl.top_k
        prev = torch.tensor(flat, dtype=torch.int32, device="cuda").reshape(wl.tokens, wl.top_k)
    st.model.layer_step(0, h, kv, wl.positions, prev, None, run_prologue=True)
    got = read_ranked(st)
    want = [] if prev is None else ranking(prev.cpu().numpy())
    assert got == want, (got, want)
    if case == "ties_and_cap":
        assert want == [3, 7, 1, 12, 0, 9, 2, 4, 5, 6, 8, 10, 11, 13]
    st.model.close()
