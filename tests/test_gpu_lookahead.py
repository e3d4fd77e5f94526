"""The lookahead-decoding forward (a 2-D Jacobi window and G candidate n-grams in one tree
attention, "万字综述 10+ 种 LLM 投机采样推理加速方案" section 8.2.3) through the C-ABI: the tree
build's mask equals the oracle's mask built from the page's two rules, bit for bit; attention
matches the oracle (all rows at the small size, sampled rows at the full size); greedy
verification and compaction are bit-exact."""
import numpy as np
import pytest
import torch

import parity_util as PU
from oracle import lookahead as OL
from speculative_decoding_draft_tree_gb300 import workloads as W
from speculative_decoding_draft_tree_gb300.api import VerifyStep

pytestmark = pytest.mark.gpu


def _check_mask(w, step):
    meta = w.meta
    want = OL.lookahead_mask(meta["W"], meta["N"], meta["G"])
    T = want.shape[0]
    anc = PU.np_(step.anc_mask).view(np.uint32)
    no = PU.np_(w.node_offset)
    for r in range(w.B):
        bits = np.zeros((T, T), dtype=bool)
        for i in range(T):
            for j in range(T):
                bits[i, j] = (anc[no[r] + i, j >> 5] >> np.uint32(j & 31)) & 1
        np.testing.assert_array_equal(bits, want)
        pos = PU.np_(step.pos_id)[no[r]:no[r] + T] - int(w.prefix_len[r])
        assert pos.tolist() == [OL.position(n) for n in OL.lookahead_nodes(meta["W"], meta["N"],
                                                                            meta["G"])]


@pytest.mark.parametrize("scale", ["small", "full"])
def test_lookahead_forward(scale):
    w = W.lookahead_config(scale=scale, device="cuda")
    snap = PU.snapshot(w)
    step = VerifyStep(w)
    step.tree_build()
    torch.cuda.synchronize()
    PU.check_tree(w, step, snap)
    _check_mask(w, step)
    step.attention()
    torch.cuda.synchronize()
    rows = None
    if scale == "full":
        rng = np.random.default_rng(11)
        rows = [(int(n), int(h)) for n, h in zip(rng.integers(0, w.N, 160),
                                                 rng.integers(0, w.H_q, 160))]
    worst = PU.check_attention(w, step, snap, rows)
    assert worst < 2e-2
    step.verify()
    torch.cuda.synchronize()
    orc = PU.oracle_verify(w, snap)
    PU.check_verify(w, step, orc)
    kb = PU.cache_region(w.k_cache, w, snap, range(w.B))
    vb = PU.cache_region(w.v_cache, w, snap, range(w.B))
    step.compact()
    torch.cuda.synchronize()
    PU.check_compact(w, step, snap, kb, vb)
    # some candidate n-grams were accepted (the generator plants pool hits)
    assert PU.np_(step.n_acc).max() >= 1
