"""spec_verify_noalloc -- verification without a caller-provided workspace.

Some callers cannot allocate device memory while they serve requests (an engine that reserves
its whole memory budget at start-up, or a plugin that is handed only tensors and a stream);
this entry point runs the same kernels on a fixed scratch array inside the library.  The test
calls it twice in a row through the C ABI (the second call sees the scratch contents the first
one left) and requires results identical to spec_verify with its own workspace.  The file is
named so that pytest collects it last."""
import pytest
import torch

from speculative_decoding_draft_tree_gb300 import binding as B
from speculative_decoding_draft_tree_gb300 import workloads as W
from speculative_decoding_draft_tree_gb300.api import VerifyStep

pytestmark = pytest.mark.gpu

OUTPUTS = ("out_tokens", "out_len", "path", "n_acc", "rejections", "req_status")


def _snapshot(step):
    return {k: getattr(step, k).clone() for k in OUTPUTS}


@pytest.mark.parametrize("cid,tau", [(4, 1.0), (5, 1.0), (3, 0.0)])
def test_noalloc_matches_workspace_entry_point(cid, tau):
    w = W.make_config(cid, scale="small", device="cuda", tau=tau)
    step = VerifyStep(w)
    step.tree_build()
    step.verify()
    torch.cuda.synchronize()
    want = _snapshot(step)
    for call in range(2):
        for k in OUTPUTS:
            if k != "req_status":
                getattr(step, k).fill_(-99)
        step.tree_build()          # re-initialises req_status
        B.spec_verify_noalloc(step.ver)
        torch.cuda.synchronize()
        got = _snapshot(step)
        for k in OUTPUTS:
            assert torch.equal(got[k], want[k]), (cid, tau, call, k)


def test_noalloc_rejects_oversize_batches():
    w = W.make_config(2, scale="small", device="cuda")
    step = VerifyStep(w)
    p = step.ver
    p.N = 40000
    with pytest.raises(B.SpecError, match="UNSUPPORTED"):
        B.spec_verify_noalloc(p)
