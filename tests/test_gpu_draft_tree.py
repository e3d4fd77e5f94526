"""Building the draft tree on the GPU (EAGLE-2 leaf expansion, top-K rows, ECHO budget; C-ABI
spec_draft_* / spec_echo_select_pack) against oracle.draft_tree.

Selections are decided on fp32 scores, so the oracle is given the GPU pool's own fp32 scores
for them and must agree bit for bit: the expand list of every level and the packed trees.  The
scores themselves are compared with the fp64 oracle: the GPU forms log q = (x - M)/tau - log Z
in fp32 (subtraction, scaling and log each within a few 1e-7 absolute for |x - M| <= 40,
log Z <= 12) and adds it to the parent's fp32 score, so a child's score must lie within
1e-5 + 2^-22 |score| of its parent's score plus the fp64 log q.  Where two tokens' log q are
that close the order between them is not unique: each returned token must carry the q-th best
fp64 log q within the same bound.
"""
import numpy as np
import pytest
import torch

from oracle import draft_tree as OD
from speculative_decoding_draft_tree_gb300 import binding as B
from speculative_decoding_draft_tree_gb300 import workloads as W
from speculative_decoding_draft_tree_gb300.api import DraftTreeBuilder

pytestmark = pytest.mark.gpu


def _oracle_pool(b):
    par, tok, dep, sc, row, cnt = [x.cpu().numpy() for x in
                                   (b.parent, b.token, b.depth_, b.score, b.row, b.count)]
    pool = OD.Pool([0] * b.B)
    pool.cands = [[dict(parent=int(par[r, i]), token=int(tok[r, i]), depth=int(dep[r, i]),
                        score=float(sc[r, i]), row=int(row[r, i])) for i in range(int(cnt[r]))]
                  for r in range(b.B)]
    return pool


def _tol(score):
    return 1e-5 + 2.0 ** -22 * abs(score)


def run_loop(B_, K, D, V, dtype, tau, K_max, scales, rows_checked=None, seed=0):
    b = DraftTreeBuilder(B_, K, D, "cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    roots = torch.randint(0, V, (B_,), generator=g, device="cuda", dtype=torch.int32)
    b.init(roots)
    checked = 0
    for level in range(1, D + 1):
        before = _oracle_pool(b)
        b.expand(level)
        torch.cuda.synchronize()
        want = OD.expand_select(before, level, K)
        got = b.expand_list.cpu().numpy()
        for r in range(B_):
            lst = [int(x) for x in got[r] if x >= 0]
            assert lst == want[r], (level, r, lst, want[r])
            assert all(x == -1 for x in got[r][len(lst):])
        rows = W.draft_level_rows(B=B_, K=K, V=V, level=level, dtype=dtype, device="cuda",
                                  seed=seed + 7, scales=scales)
        b.append(level, rows, V, tau)
        torch.cuda.synchronize()
        after = _oracle_pool(b)
        rows_np = rows[:, :V].float().cpu().numpy()
        for r in range(B_):
            base = len(before.cands[r])
            assert len(after.cands[r]) == base + len(want[r]) * K
            for j, cand in enumerate(want[r]):
                assert after.cands[r][cand]["row"] == (level - 1) * B_ * K + r * K + j
                kids = after.cands[r][base + j * K: base + (j + 1) * K]
                assert all(k["parent"] == cand and k["depth"] == level for k in kids)
                if rows_checked is not None and (r * K + j) % rows_checked:
                    continue
                checked += 1
                lq = OD.log_softmax(rows_np[r * K + j], tau)
                toks, lps = OD.topk(rows_np[r * K + j], K, tau)
                gt = [k["token"] for k in kids]
                assert len(set(gt)) == K
                psc = after.cands[r][cand]["score"]
                for q, k in enumerate(kids):
                    assert abs(lq[k["token"]] - lps[q]) <= _tol(k["score"]), (level, r, j, q)
                    assert abs(k["score"] - (psc + lq[k["token"]])) <= _tol(k["score"])
    assert checked > 0
    b.echo(K_max)
    torch.cuda.synchronize()
    final = _oracle_pool(b)
    kept = OD.echo_select(final, K_max)
    want = OD.pack(final, kept)
    got = b.packed()
    np.testing.assert_array_equal(got["node_offset"].cpu().numpy(), want["node_offset"])
    for key in ("parent", "tokens", "depth", "draft_row"):
        np.testing.assert_array_equal(got[key].cpu().numpy(), want[key], err_msg=key)
    np.testing.assert_array_equal(got["source"].cpu().numpy(), [i for _, i in want["source"]])
    # the packed trees are what the verification step reads: the tree build accepts them
    no = got["node_offset"]
    N = int(no[-1])
    T_max = int((no[1:] - no[:-1]).max())
    i32 = dict(dtype=torch.int32, device="cuda")
    st = torch.zeros(B_, **i32)
    depth = torch.empty(N, **i32)
    pos = torch.empty(N, **i32)
    anc = torch.empty((N, (T_max + 31) // 32), **i32)
    internal = torch.empty(N, dtype=torch.uint8, device="cuda")
    B.spec_tree_build(got["parent"].contiguous(), no, torch.zeros(B_, **i32), T_max, depth, pos,
                      anc, internal, st)
    torch.cuda.synchronize()
    assert not st.cpu().numpy().any()
    np.testing.assert_array_equal(depth.cpu().numpy(), want["depth"])
    return b, final, kept


@pytest.mark.parametrize("dtype,tau", [("bf16", 1.0), ("f32", 1.0), ("bf16", 0.6)])
def test_draft_tree_small(dtype, tau):
    run_loop(B_=5, K=3, D=5, V=3001, dtype=dtype, tau=tau, K_max=60,
             scales=[4.0, 0.5, 1.0, 2.0, 0.3])


def test_draft_tree_budget_edges():
    # a budget below the roots keeps only the roots; a huge one keeps every candidate
    for K_max, want_total in ((3, 4), (10 ** 6, None)):
        b, final, kept = run_loop(B_=4, K=2, D=3, V=517, dtype="bf16", tau=1.0, K_max=K_max,
                                  scales=[1.0, 2.0, 3.0, 0.5])
        total = int(b.node_offset[-1])
        assert total == (want_total if want_total else sum(len(c) for c in final.cands))


def test_draft_tree_full_size():
    """The EAGLE-2 / ECHO workload's shape: 64 requests, top-5 expansion to depth 8, vocab
    152064, K_max 2048 (row values checked on every 32nd expanded row)."""
    rng = np.random.default_rng(3)
    scales = rng.uniform(0.3, 4.0, size=64).tolist()
    b, final, kept = run_loop(B_=64, K=5, D=8, V=152064, dtype="bf16", tau=1.0, K_max=2048,
                              scales=scales, rows_checked=32)
    assert int(b.node_offset[-1]) == 2048
