"""Building the draft tree on the GPU (EAGLE-2 leaf expansion, top-K rows, ECHO budget; C-ABI
spec_draft_* / spec_echo_select_pack) against oracle.draft_tree.build, run independently.

Both sides start from the same seeded inputs only (root tokens and the draft model's rows of
every level); the oracle builds the whole tree in fp64 on its own and nothing it reads comes
from a GPU buffer.  Compared: every level's expand list, every candidate's token, parent, depth,
row and score, and the packed trees, bit for bit except the scores.

Score bound: the GPU forms log q = (x - M)/tau - log Z in fp32 (subtraction, scaling and log
each within a few 1e-7 absolute for |x - M| <= 40, log Z <= 12, so under 1e-5 per level) and
adds it to the parent's fp32 score (one rounding, 2^-24 relative), so a depth-d candidate's score
lies within d (1e-5 + 2^-24 |score|) of the fp64 path sum.

Selections are decided on those fp32 scores, so a decision whose two fp64 sides lie within the
sum of their bounds has no unique answer: such near ties (a top-K boundary or the order inside
a top-K list, the K-best cut of a level's frontier, ECHO's budget cut) are found on the oracle
side, and only requests touched by one may differ from the oracle; they are counted and
reported (the tally is printed and must stay below 1% of requests).  Exactly equal values tie
the same way on both sides (lower token id / candidate index / request)."""
import numpy as np
import pytest
import torch

from oracle import draft_tree as OD
from speculative_decoding_draft_tree_gb300 import binding as B
from speculative_decoding_draft_tree_gb300 import workloads as W
from speculative_decoding_draft_tree_gb300.api import DraftTreeBuilder

pytestmark = pytest.mark.gpu

TALLY = {"requests": 0, "exempt": 0}


def _tol(score, depth):
    return max(depth, 1) * (1e-5 + 2.0 ** -24 * abs(score))


def _gpu_pool(b):
    par, tok, dep, sc, row, cnt = [x.cpu().numpy() for x in
                                   (b.parent, b.token, b.depth_, b.score, b.row, b.count)]
    return [[dict(parent=int(par[r, i]), token=int(tok[r, i]), depth=int(dep[r, i]),
                  score=float(sc[r, i]), row=int(row[r, i])) for i in range(int(cnt[r]))]
            for r in range(b.B)]


def _near_ties(pool, chosen_log, rows_np, K, tau, K_max):
    """Requests whose construction passes a decision that fp32 cannot settle uniquely."""
    B_ = pool.B
    touched = set()
    for level, chosen in chosen_log.items():
        for r in range(B_):
            cs = pool.cands[r]
            if level > 1:
                front = sorted(([cs[i]["score"], i] for i in range(len(cs))
                                if cs[i]["depth"] == level - 1), key=lambda x: (-x[0], x[1]))
                if len(front) > K:
                    a, c = front[K - 1][0], front[K][0]
                    if a != c and a - c <= 2 * _tol(a, level - 1):
                        touched.add(r)
            for j in range(len(chosen[r])):
                lq = OD.log_softmax(rows_np[level - 1][r * K + j], tau)
                top = np.sort(lq)[::-1][:K + 1]
                d = top[:-1] - top[1:]
                if np.any((d > 0) & (d <= 2e-5)):
                    touched.add(r)
    nonroot = sorted(((c["score"], r, i) for r, cs in enumerate(pool.cands)
                      for i, c in enumerate(cs) if i > 0), key=lambda x: (-x[0], x[1], x[2]))
    cut = K_max - B_
    if 0 < cut < len(nonroot):
        edge = nonroot[cut - 1][0]
        for s, r, i in nonroot:
            if abs(s - edge) <= 2 * _tol(edge, pool.cands[r][i]["depth"]) and s != edge:
                touched.add(r)
                touched.add(nonroot[cut - 1][1])
    return touched


def run_independent(B_, K, D, V, dtype, tau, K_max, scales, seed=0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    roots = torch.randint(0, V, (B_,), generator=g, device="cuda", dtype=torch.int32)
    rows = [W.draft_level_rows(B=B_, K=K, V=V, level=lv, dtype=dtype, device="cuda",
                               seed=seed + 7, scales=scales) for lv in range(1, D + 1)]
    # inputs of both sides, copied to the host before any kernel of the library runs
    roots_np = roots.cpu().numpy()
    rows_np = [r[:, :V].float().cpu().numpy() for r in rows]

    # the oracle, alone
    chosen_log = {}

    def rows_of_level(level, chosen):
        chosen_log[level] = [list(c) for c in chosen]
        row_ids = [[(level - 1) * B_ * K + r * K + j for j in range(len(chosen[r]))]
                   for r in range(B_)]
        rws = [[rows_np[level - 1][r * K + j] for j in range(len(chosen[r]))] for r in range(B_)]
        return row_ids, rws

    pool, kept, want = OD.build(roots_np, rows_of_level, K, D, K_max, tau)

    # the GPU
    b = DraftTreeBuilder(B_, K, D, "cuda")
    b.init(roots)
    gpu_expand = {}
    for level in range(1, D + 1):
        b.expand(level)
        gpu_expand[level] = b.expand_list.cpu().numpy().copy()
        b.append(level, rows[level - 1], V, tau)
    b.echo(K_max)
    torch.cuda.synchronize()
    gpool = _gpu_pool(b)
    got = b.packed()

    touched = _near_ties(pool, chosen_log, rows_np, K, tau, K_max)
    differ = set()
    for r in range(B_):
        ok = True
        for level, chosen in chosen_log.items():
            lst = [int(x) for x in gpu_expand[level][r] if x >= 0]
            ok &= lst == chosen[r] and all(x == -1 for x in gpu_expand[level][r][len(lst):])
        oc, gc = pool.cands[r], gpool[r]
        ok &= len(oc) == len(gc)
        if ok:
            for i, (o, c) in enumerate(zip(oc, gc)):
                ok &= (o["parent"], o["token"], o["depth"], o["row"]) == \
                      (c["parent"], c["token"], c["depth"], c["row"])
                ok &= abs(o["score"] - c["score"]) <= _tol(o["score"], o["depth"])
        if not ok:
            differ.add(r)
    # packed trees: request by request
    gno = got["node_offset"].cpu().numpy()
    keys = ("parent", "tokens", "depth", "draft_row")
    gp = {k: got[k].cpu().numpy() for k in keys}
    gsrc = got["source"].cpu().numpy()
    for r in range(B_):
        a0, a1, b0, b1 = want["node_offset"][r], want["node_offset"][r + 1], gno[r], gno[r + 1]
        same = (a1 - a0) == (b1 - b0) and all(np.array_equal(want[k][a0:a1], gp[k][b0:b1])
                                              for k in keys)
        same = same and [i for rr, i in want["source"][a0:a1]] == gsrc[b0:b1].tolist()
        if not same:
            differ.add(r)
    unexplained = differ - touched
    assert not unexplained, f"requests differing from the oracle without a near tie: {sorted(unexplained)}"
    TALLY["requests"] += B_
    TALLY["exempt"] += len(differ)
    print(f"draft tree B={B_} V={V}: {len(differ)} of {B_} requests differ at near ties "
          f"({len(touched)} touched by one)")
    assert len(differ) <= max(1, B_ // 100)
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
    np.testing.assert_array_equal(depth.cpu().numpy(), gp["depth"])
    return b, pool, want


@pytest.mark.parametrize("dtype,tau", [("bf16", 1.0), ("f32", 1.0), ("bf16", 0.6)])
def test_draft_tree_small(dtype, tau):
    run_independent(B_=5, K=3, D=5, V=3001, dtype=dtype, tau=tau, K_max=60,
                    scales=[4.0, 0.5, 1.0, 2.0, 0.3])


def test_draft_tree_budget_edges():
    # a budget below the roots keeps only the roots; a huge one keeps every candidate
    for K_max, want_total in ((3, 4), (10 ** 6, None)):
        b, pool, want = run_independent(B_=4, K=2, D=3, V=517, dtype="bf16", tau=1.0,
                                        K_max=K_max, scales=[1.0, 2.0, 3.0, 0.5])
        total = int(b.node_offset[-1])
        assert total == (want_total if want_total else sum(len(c) for c in pool.cands))


def test_draft_tree_full_size():
    """The EAGLE-2 / ECHO workload's shape: 64 requests, top-5 expansion to depth 8, vocab
    152064, K_max 2048; every candidate's score checked."""
    rng = np.random.default_rng(3)
    scales = rng.uniform(0.3, 4.0, size=64).tolist()
    b, pool, want = run_independent(B_=64, K=5, D=8, V=152064, dtype="bf16", tau=1.0,
                                    K_max=2048, scales=scales)
    assert int(b.node_offset[-1]) == 2048
