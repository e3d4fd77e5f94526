"""Parity at the full workload sizes, in the launch configuration the benchmark uses: every
request for the tree, verification and compaction outputs (bit-exact), and sampled
(node, head) rows for attention (2e-2 absolute for bf16) -- the oracle computes those rows one by
one over the request's whole KV range.  The chain and Medusa workloads run at tau = 1 and
tau = 0 (greedy), the chain also at draft noise sigma = 0.5 and 2 (high and low acceptance)."""
import numpy as np
import pytest
import torch

import parity_util as PU
from speculative_decoding_draft_tree_gb300 import workloads as W
from speculative_decoding_draft_tree_gb300.api import VerifyStep

pytestmark = pytest.mark.gpu


def _sample_rows(w, snap, n_req, seed):
    rng = np.random.default_rng(seed)
    no = snap["node_offset"]
    reqs = sorted(rng.choice(w.B, size=min(n_req, w.B), replace=False).tolist())
    rows = []
    for r in reqs:
        o, T = int(no[r]), int(no[r + 1] - no[r])
        nodes = sorted({o, o + T - 1, o + int(rng.integers(0, T))})
        heads = sorted({0, w.H_q - 1, int(rng.integers(0, w.H_q))})
        rows += [(n, h) for n in nodes for h in heads]
    return rows


CASES = [(2, 16, 1.0, 1.0), (2, 4, 0.0, 1.0), (2, 4, 1.0, 0.5), (2, 4, 1.0, 2.0),
         (3, 4, 1.0, 1.0), (3, 2, 0.0, 1.0), (4, 8, 1.0, 1.0), (5, 10, 1.0, 1.0)]


@pytest.mark.parametrize("cid,n_req,tau,sigma", CASES)
def test_full_size_parity(cid, n_req, tau, sigma):
    w = W.make_config(cid, scale="full", device="cuda", tau=tau, sigma=sigma)
    snap = PU.snapshot(w)
    step = VerifyStep(w)
    step.tree_build()
    step.attention()
    torch.cuda.synchronize()
    PU.check_tree(w, step, snap)
    assert (PU.np_(step.req_status) == 0).all()
    worst = PU.check_attention(w, step, snap, _sample_rows(w, snap, n_req, seed=cid))
    step.verify()
    torch.cuda.synchronize()
    orc = PU.oracle_verify(w, snap)
    draws, exempt = PU.check_verify(w, step, orc)
    kb = PU.cache_region(w.k_cache, w, snap, range(w.B))
    vb = PU.cache_region(w.v_cache, w, snap, range(w.B))
    step.compact()
    torch.cuda.synchronize()
    PU.check_compact(w, step, snap, kb, vb)
    print(f"config {cid} tau {tau} sigma {sigma}: attention max |err| {worst:.3g}, verify draws "
          f"{draws}, near-boundary exemptions {exempt}")
