"""Multi-draft verification (siblings proposed by different draft models, each child with its
own q row; the running residual applied sibling after sibling) through the C-ABI against the
oracle's SIBLING_MULTI_DRAFT rule: bit-exact tokens, paths and rejection counts (up to the
1e-6 guard band), and compaction after it."""
import numpy as np
import pytest
import torch

import parity_util as PU
from oracle import verify as OV
from speculative_decoding_draft_tree_gb300 import binding as B
from speculative_decoding_draft_tree_gb300 import workloads as W
from speculative_decoding_draft_tree_gb300.api import VerifyStep

pytestmark = pytest.mark.gpu


def _run(w):
    snap = PU.snapshot(w)
    step = VerifyStep(w, sibling_rule=B.SPEC_SIBLING_MULTI_DRAFT)
    step.tree_build()
    step.verify()
    torch.cuda.synchronize()
    orc = PU.oracle_verify(w, snap, OV.SIBLING_MULTI_DRAFT)
    draws, exempt = PU.check_verify(w, step, orc)
    kb = PU.cache_region(w.k_cache, w, snap, range(w.B))
    vb = PU.cache_region(w.v_cache, w, snap, range(w.B))
    step.compact()
    torch.cuda.synchronize()
    PU.check_compact(w, step, snap, kb, vb)
    return step, orc


@pytest.mark.parametrize("tau,kind", [(1.0, W.DRAFT_LOGITS), (0.7, W.DRAFT_LOGITS),
                                      (1.0, W.DRAFT_PROBS), (1.6, W.DRAFT_PROBS)])
def test_multidraft_small(tau, kind):
    total_rej = 0
    for seed in range(4):
        w = W.multidraft_workload(B=4, k=4, gamma=2, V=2999, dtype="bf16", H_q=4, H_kv=2, d=128,
                                  prefix=[40, 301, 7, 16], tau=tau, noise_stds=[2.0, 2.5, 3.0, 3.5],
                                  device="cuda", draft_kind=kind,
                                  seeds=dict(logits=100 + seed, drafting=200 + seed,
                                             uniform=seed))
        step, orc = _run(w)
        total_rej += int(np.asarray(orc["rejections"]).sum())
    assert total_rej >= 8   # rejected siblings exercised the residual passes


def test_multidraft_greedy():
    w = W.multidraft_config(scale="small", device="cuda", tau=0.0)
    _run(w)


def test_multidraft_full():
    w = W.multidraft_config(scale="full", device="cuda")
    step, orc = _run(w)
    assert int(np.asarray(orc["rejections"]).sum()) > 0


def test_multidraft_f32_logits():
    w = W.multidraft_workload(B=3, k=3, gamma=2, V=1001, dtype="f32", H_q=4, H_kv=4, d=64,
                              prefix=33, tau=1.0, noise_stds=[2.0, 3.0, 4.0], device="cuda")
    _run(w)


def test_shared_rows_named_per_child():
    """A SpecInfer tree (top-k siblings from one shared row) with the row named per child: the
    multi-draft rule on the GPU against the oracle's."""
    w = W.make_config(4, scale="small", device="cuda")
    par = w.parent.cpu().numpy()
    no = w.node_offset.cpu().numpy()
    dr = w.draft_row.cpu().numpy()
    per_child = np.full_like(dr, -1)
    for r in range(w.B):
        for c in range(1, no[r + 1] - no[r]):
            per_child[no[r] + c] = dr[no[r] + par[no[r] + c]]
    w.draft_row.copy_(torch.as_tensor(per_child, device="cuda"))
    _run(w)
