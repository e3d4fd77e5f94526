"""Failure detection on the GPU without a fault: a bounded device wait is made to run out (a wait
for a device flag that nothing sets, through the library's testing hook) and the call must report
it in the request status, keep its outputs well-formed, finish in bounded time, and leave the
context usable for the next call."""
import time

import numpy as np
import pytest
import torch

from oracle import draft_tree as OD
from speculative_decoding_draft_tree_gb300 import binding as B
from speculative_decoding_draft_tree_gb300 import workloads as W
from speculative_decoding_draft_tree_gb300.api import DraftTreeBuilder

pytestmark = pytest.mark.gpu


def test_expired_wait_times_out_and_the_context_stays_usable():
    Bn, K, V = 4, 3, 3001
    roots = torch.arange(Bn, dtype=torch.int32, device="cuda") * 7
    rows = W.draft_level_rows(B=Bn, K=K, V=V, level=1, device="cuda", scales=[1.0, 2.0, 0.5, 3.0])
    b = DraftTreeBuilder(Bn, K, 3, "cuda")
    b.init(roots)
    b.expand(1)
    B.spec_debug_draft_copy_stall(0)
    try:
        t0 = time.time()
        b.append(1, rows, V)
        torch.cuda.synchronize()
        elapsed = time.time() - t0
    finally:
        B.spec_debug_draft_copy_stall(-1)
    assert elapsed < 30.0
    st = b.req_status.cpu().numpy()
    assert ((st & B.REQ_BITS["TIMEOUT"]) != 0).all()
    tok = b.token.cpu().numpy()
    score = b.score.cpu().numpy()
    assert (tok[:, 1:1 + K] == -1).all() and np.isneginf(score[:, 1:1 + K]).all()

    # the same construction again, hook off: status clean, children = the row's top-K
    b.init(roots)
    b.expand(1)
    b.append(1, rows, V)
    torch.cuda.synchronize()
    assert not b.req_status.cpu().numpy().any()
    rows_np = rows[:, :V].float().cpu().numpy()
    tok = b.token.cpu().numpy()
    for r in range(Bn):
        want, _ = OD.topk(rows_np[r * K], K)
        lq = OD.log_softmax(rows_np[r * K])
        got = tok[r, 1:1 + K]
        # the same tokens unless two log-probabilities tie within fp32 resolution
        assert np.allclose(lq[got], lq[want], atol=1e-5)
