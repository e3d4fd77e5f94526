"""spec_verify_noalloc -- verification without a caller-provided workspace.

Some callers cannot allocate device memory while they serve requests (an engine that reserves
its whole memory budget at start-up, or a plugin that is handed only tensors and a stream);
this entry point runs the same kernels on a fixed scratch array inside the library.  The test
calls it twice in a row through the C ABI, each time right after a call on a different
workload (other vocabulary, tree and row count) that leaves its own statistics in the shared
array, and requires results identical to spec_verify with its own workspace.  The file is
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


CASES = [(4, 1.0, "auto"), (5, 1.0, "auto"), (3, 0.0, "auto"), (2, 1.0, "split"),
         (4, 1.0, "walk"), (3, 0.0, "walk")]
PATHS = {"auto": B.SPEC_VERIFY_PATH_AUTO, "split": B.SPEC_VERIFY_PATH_SPLIT,
         "walk": B.SPEC_VERIFY_PATH_WALK}


@pytest.mark.parametrize("cid,tau,path", CASES)
def test_noalloc_matches_workspace_entry_point(cid, tau, path):
    w = W.make_config(cid, scale="small", device="cuda", tau=tau)
    step = VerifyStep(w, verify_path=PATHS[path])
    step.tree_build()
    step.verify()
    torch.cuda.synchronize()
    want = _snapshot(step)
    # another workload whose calls fill the shared array with statistics of other rows
    other = VerifyStep(W.make_config(5 if cid != 5 else 4, scale="small", device="cuda"),
                       verify_path=B.SPEC_VERIFY_PATH_SPLIT)
    other.tree_build()
    for call in range(2):
        B.spec_verify_noalloc(other.ver)
        for k in OUTPUTS:
            if k != "req_status":
                getattr(step, k).fill_(-99)
        step.tree_build()          # re-initialises req_status
        B.spec_verify_noalloc(step.ver)
        torch.cuda.synchronize()
        got = _snapshot(step)
        for k in OUTPUTS:
            assert torch.equal(got[k], want[k]), (cid, tau, path, call, k)


def test_noalloc_refuses_multi_draft():
    # the multi-draft rule keeps residual rows per request, which the fixed array does not hold
    w = W.multidraft_config(scale="small", device="cuda")
    step = VerifyStep(w, sibling_rule=B.SPEC_SIBLING_MULTI_DRAFT)
    with pytest.raises(B.SpecError, match="UNSUPPORTED"):
        B.spec_verify_noalloc(step.ver)


def test_noalloc_rejects_oversize_batches():
    w = W.make_config(2, scale="small", device="cuda")
    step = VerifyStep(w)
    p = step.ver
    p.N = 40000
    with pytest.raises(B.SpecError, match="UNSUPPORTED"):
        B.spec_verify_noalloc(p)
