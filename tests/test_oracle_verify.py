"""Pins for oracle.verify.

* E[L] = (1 - a^(g+1)) / (1 - a) for a chain of g drafts whose per-position acceptance rate is
  a = sum_x min(p, q) = 1 - TV(p, q) ("【模型后训练与深度推理】9 推理加速：推测解码与级联推理" 7.2), by Monte
  Carlo over 10^5 rounds, +-1%.
* Losslessness (the emitted tokens follow p; "推测解码 2026" and section 7.1 of the CSDN page),
  checked EXACTLY: the law of the oracle's output is integrated over every draft assignment and,
  by bisection on the oracle's own accept / reject and sampling decisions (black box: only its
  outputs are observed), over the uniforms; the first emitted token must follow p_root to 1e-9
  and every later one, given the accepted tokens before it, p(. | those tokens) to 1e-8, down
  to the bonus token after a fully accepted path.
* The same losslessness by chi-square on vocab 16 with several iid siblings.
* Multi-draft siblings (each child drawn from its own small model's q): the same exact
  losslessness, and agreement with the closed-form residual rule when every sibling's q is the
  same.
* Greedy: with greedy drafts, tau -> 0+ sampling reproduces the tau = 0 argmax walk.
"""
from collections import defaultdict
from itertools import product

import numpy as np
import pytest
import torch

from oracle import verify as OV


# ----------------------------------------------------------------------------------------------
# helpers building explicit small cases
# ----------------------------------------------------------------------------------------------
def _dist(rng, V, conc=1.0):
    return rng.dirichlet(np.full(V, conc))


def _run(case, u_acc, u_samp, rule):
    T = len(case["parent"])
    uni = np.stack([u_acc, u_samp], axis=1)
    res = OV.verify(case["target"], case["draft"], case["kind"], case["draft_row"],
                    case["tokens"], case["parent"], [0, T], uni, case["tau"], case["V"],
                    max_path=T, sibling_rule=rule, T_max=T)
    assert res["status"][0] == 0
    return tuple(res["out_tokens"][0]), res["path"][0], res["events"][0]


_ONE_MINUS = np.nextafter(1.0, 0.0)


def _bracket(pred, iters=44):
    """pred(u) is True on [0, t) and False on [t, 1); return (lo, hi) with pred(lo) True,
    pred(hi) False and hi - lo <= 2^-iters (hi = 1.0 when pred never fails)."""
    if not pred(0.0):
        return 0.0, 0.0
    if pred(_ONE_MINUS):
        return 1.0, 1.0
    lo, hi = 0.0, 1.0
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if pred(mid):
            lo = mid
        else:
            hi = mid
    return lo, hi


def _threshold(pred, iters=44):
    lo, hi = _bracket(pred, iters)
    return 0.5 * (lo + hi)


def _exact_law(case, rule):
    """Law of the emitted sequence over the uniforms (draft tokens fixed in `case`)."""
    T = len(case["parent"])
    law = defaultdict(float)

    def rec(fixed, weight):
        u_acc = np.array([fixed.get(i, 0.5) for i in range(T)])
        _, path, events = _run(case, u_acc, np.full(T, 0.5), rule)
        pending = [e[2] for e in events if e[0] == "test" and e[2] not in fixed]
        if pending:
            c = pending[0]

            def accepted(u):
                ua = u_acc.copy()
                ua[c] = u
                return c in _run(case, ua, np.full(T, 0.5), rule)[1]

            t = _threshold(accepted)
            if t > 0:
                rec({**fixed, c: 0.5 * t}, weight * t)
            if t < 1:
                rec({**fixed, c: 0.5 * (1 + t)}, weight * (1 - t))
            return
        stop = path[-1]

        def final(u):
            us = np.full(T, 0.5)
            us[stop] = u
            return _run(case, u_acc, us, rule)[0]

        start, seq = 0.0, final(0.0)
        while True:     # the final token is monotone in u_samp: walk its steps left to right
            if final(_ONE_MINUS) == seq:
                law[seq] += weight * (1.0 - start)
                break
            lo, hi = _bracket(lambda u: u < start or final(u) == seq)
            mid = 0.5 * (lo + hi)
            law[seq] += weight * (mid - start)
            start, seq = mid, final(hi)

    rec({}, 1.0)
    return law


def _tree_case(V, tau, kind, shape, rng):
    """Contexts: every node's target / draft row is a function of its path's tokens, as for a
    real model.  shape: parent array.  Returns a factory mapping draft tokens -> case."""
    T = len(shape)
    tables_t, tables_q = {}, {}

    def rows(ctx):
        if ctx not in tables_t:
            tables_t[ctx] = rng.normal(size=V) * 1.5
            tables_q[ctx] = rng.normal(size=V) * 1.5
        return tables_t[ctx], tables_q[ctx]

    def make(draft_tokens):
        tokens = [0] + list(draft_tokens)
        ctx = [()] * T
        for i in range(1, T):
            ctx[i] = ctx[shape[i]] + (tokens[i],)
        tgt = np.stack([rows(ctx[i])[0] for i in range(T)])
        drl = np.stack([rows(ctx[i])[1] for i in range(T)])
        if kind == OV.DRAFT_PROBS:
            drl = np.stack([OV.softmax_at(x, 1.0) for x in drl])
        return dict(target=tgt, draft=drl, kind=kind, draft_row=np.arange(T), tokens=tokens,
                    parent=shape, tau=tau, V=V, ctx=ctx)

    return make, rows


def _q_of(case, node):
    row = case["draft"][node]
    return OV.softmax_at(row, case["tau"]) if case["kind"] == OV.DRAFT_LOGITS else row


def _p_of(rows, ctx, tau):
    return torch.softmax(torch.tensor(rows(ctx)[0]) / tau, dim=0).numpy()


def _assert_every_token_follows_p(total, rows, tau, V):
    """The emitted tokens follow the target model: the first one p_root, and every later one,
    given the tokens before it (accepted drafts, since a token follows them), p(. | those
    tokens) -- down to the bonus token after a fully accepted path."""
    first = np.zeros(V)
    for seq, pr in total.items():
        first[seq[0]] += pr
    np.testing.assert_allclose(first, _p_of(rows, (), tau), atol=1e-9)
    by_prefix = defaultdict(lambda: np.zeros(V))
    for seq, pr in total.items():
        for k in range(1, len(seq)):
            by_prefix[seq[:k]][seq[k]] += pr
    assert by_prefix
    for prefix, cond in by_prefix.items():
        if cond.sum() > 1e-4:
            np.testing.assert_allclose(cond / cond.sum(), _p_of(rows, prefix, tau), atol=1e-8)


@pytest.mark.parametrize("shape,V,tau,kind", [
    ([-1, 0, 0, 0], 3, 1.0, OV.DRAFT_LOGITS),      # three iid siblings at the root
    ([-1, 0, 0, 1], 3, 0.7, OV.DRAFT_PROBS),       # two siblings, the first one has a child
    ([-1, 0, 1], 4, 1.3, OV.DRAFT_LOGITS),         # chain of two drafts
])
def test_exact_losslessness(shape, V, tau, kind):
    rng = np.random.default_rng(11)
    make, rows = _tree_case(V, tau, kind, shape, rng)
    T = len(shape)
    total = defaultdict(float)
    probe = make([0] * (T - 1))
    for draft in product(range(V), repeat=T - 1):
        case = make(draft)
        w = 1.0
        for c in range(1, T):   # node c was drawn from q of its parent
            w *= _q_of(case, shape[c])[draft[c - 1]]
        for seq, pr in _exact_law(case, OV.SIBLING_RESIDUAL).items():
            total[seq] += w * pr
    assert abs(sum(total.values()) - 1.0) < 1e-9
    _assert_every_token_follows_p(total, rows, tau, V)
    del probe


def _multi_case(V, tau, kind, shape, rng):
    """Like _tree_case, but child c is drawn from draft model k = its rank among its siblings,
    with model k's own q in every context; draft row c holds the q child c was drawn from."""
    T = len(shape)
    tables_t, tables_q = {}, {}

    def rows(ctx):
        if ctx not in tables_t:
            tables_t[ctx] = rng.normal(size=V) * 1.5
        return tables_t[ctx], None

    def qrow(ctx, k):
        if (ctx, k) not in tables_q:
            tables_q[(ctx, k)] = rng.normal(size=V) * 1.5
        return tables_q[(ctx, k)]

    rank = [0] * T
    for c in range(1, T):
        rank[c] = sum(1 for j in range(1, c) if shape[j] == shape[c])

    def make(draft_tokens):
        tokens = [0] + list(draft_tokens)
        ctx = [()] * T
        for i in range(1, T):
            ctx[i] = ctx[shape[i]] + (tokens[i],)
        tgt = np.stack([rows(ctx[i])[0] for i in range(T)])
        drl = np.stack([np.zeros(V)] + [qrow(ctx[shape[c]], rank[c]) for c in range(1, T)])
        if kind == OV.DRAFT_PROBS:
            drl = np.stack([OV.softmax_at(x, 1.0) for x in drl])
        return dict(target=tgt, draft=drl, kind=kind, draft_row=np.arange(T), tokens=tokens,
                    parent=shape, tau=tau, V=V, ctx=ctx)

    return make, rows


@pytest.mark.parametrize("shape,V,tau,kind", [
    ([-1, 0, 0, 0], 3, 1.0, OV.DRAFT_LOGITS),      # three siblings from three draft models
    ([-1, 0, 0, 1], 3, 0.7, OV.DRAFT_PROBS),       # two models at the root, then one deeper
])
def test_exact_losslessness_multi_draft(shape, V, tau, kind):
    rng = np.random.default_rng(12)
    make, rows = _multi_case(V, tau, kind, shape, rng)
    T = len(shape)
    total = defaultdict(float)
    for draft in product(range(V), repeat=T - 1):
        case = make(draft)
        w = 1.0
        for c in range(1, T):   # node c was drawn from its own row's q
            w *= _q_of(case, c)[draft[c - 1]]
        for seq, pr in _exact_law(case, OV.SIBLING_MULTI_DRAFT).items():
            total[seq] += w * pr
    assert abs(sum(total.values()) - 1.0) < 1e-9
    _assert_every_token_follows_p(total, rows, tau, V)


def test_multi_draft_with_one_q_equals_the_closed_form():
    """When every sibling was drawn from the same q, the sequential residual is the closed-form
    k-fold residual: both rules take the same decisions on the same uniforms."""
    rng = np.random.default_rng(13)
    V, shape = 40, [-1, 0, 0, 0, 0, 1, 1, 2]
    T = len(shape)
    for trial in range(60):
        tgt = rng.normal(size=(T, V)) * 2.0
        q_parent = rng.normal(size=(T, V)) * 2.0
        tokens = [0] + [int(x) for x in rng.integers(0, V, T - 1)]
        uni = rng.random((T, 2))
        # per-parent rows for the residual rule, the same rows named per child for multi-draft
        per_child = np.array([0] + [shape[c] for c in range(1, T)])
        a = OV.verify(tgt, q_parent, OV.DRAFT_LOGITS, np.arange(T), tokens, shape, [0, T], uni,
                      1.0, V, T, sibling_rule=OV.SIBLING_RESIDUAL, T_max=T)
        b = OV.verify(tgt, q_parent, OV.DRAFT_LOGITS, per_child, tokens, shape, [0, T], uni,
                      1.0, V, T, sibling_rule=OV.SIBLING_MULTI_DRAFT, T_max=T)
        assert a["out_tokens"] == b["out_tokens"] and a["rejections"].tolist() == b["rejections"].tolist()


@pytest.mark.parametrize("kind", [OV.DRAFT_LOGITS, OV.DRAFT_PROBS])
def test_independent_rule_is_lossless_on_chains(kind):
    """With one child per node the per-sibling p/q test and its resampling from
    norm(max(0, p - q)) are plain speculative sampling: the exact law follows p."""
    rng = np.random.default_rng(14)
    shape, V, tau = [-1, 0, 1], 4, 0.8
    make, rows = _tree_case(V, tau, kind, shape, rng)
    total = defaultdict(float)
    for draft in product(range(V), repeat=2):
        case = make(draft)
        w = _q_of(case, 0)[draft[0]] * _q_of(case, 1)[draft[1]]
        for seq, pr in _exact_law(case, OV.SIBLING_INDEPENDENT).items():
            total[seq] += w * pr
    assert abs(sum(total.values()) - 1.0) < 1e-9
    _assert_every_token_follows_p(total, rows, tau, V)


def test_independent_sibling_rule_is_biased():
    """The literal per-sibling p/q test (every sibling against the original p) is not lossless
    for several iid siblings: the exact law of the first token moves away from p."""
    rng = np.random.default_rng(5)
    shape, V, tau = [-1, 0, 0, 0], 3, 1.0
    make, rows = _tree_case(V, tau, OV.DRAFT_LOGITS, shape, rng)
    first = np.zeros(V)
    for draft in product(range(V), repeat=3):
        case = make(draft)
        w = np.prod([_q_of(case, 0)[t] for t in draft])
        for seq, pr in _exact_law(case, OV.SIBLING_INDEPENDENT).items():
            first[seq[0]] += w * pr
    assert np.abs(first - _p_of(rows, (), tau)).max() > 1e-3


# ----------------------------------------------------------------------------------------------
# Monte Carlo pins
# ----------------------------------------------------------------------------------------------
def _pq_with_alpha(rng, V, alpha):
    p = _dist(rng, V)
    r = _dist(rng, V, 0.3)

    def acc(t):
        return np.minimum(p, (1 - t) * p + t * r).sum()

    lo, hi = 0.0, 1.0
    assert acc(1.0) < alpha
    for _ in range(100):
        mid = 0.5 * (lo + hi)
        if acc(mid) > alpha:
            lo = mid
        else:
            hi = mid
    q = (1 - lo) * p + lo * r
    return p, q / q.sum(), np.minimum(p, q / q.sum()).sum()


@pytest.mark.parametrize("gamma,alpha", [(1, 0.2), (4, 0.5), (8, 0.8), (5, 0.95)])
def test_expected_emitted_length(gamma, alpha):
    rng = np.random.default_rng(100 + gamma)
    V, rounds = 16, 100_000
    p, q, a = _pq_with_alpha(rng, V, alpha)
    T = gamma + 1
    B = rounds
    parent = np.tile(np.array([-1] + list(range(gamma))), B)
    no = np.arange(B + 1) * T
    tgt = np.tile(np.log(p), (B * T, 1))
    drf = q[None, :]
    drow = np.zeros(B * T, dtype=np.int64)
    cdf = np.cumsum(q)
    tokens = np.minimum(np.searchsorted(cdf, rng.random(B * T) * cdf[-1], side="right"), V - 1)
    uni = rng.random((B * T, 2))
    res = OV.verify(tgt, drf, OV.DRAFT_PROBS, drow, tokens, parent, no, uni, 1.0, V,
                    max_path=T, T_max=T)
    mean_L = res["out_len"].mean()
    want = (1 - a ** (gamma + 1)) / (1 - a)
    assert abs(mean_L - want) / want < 0.01, (mean_L, want, a)


def test_chi_square_first_token_follows_p():
    from scipy.stats import chisquare
    rng = np.random.default_rng(7)
    V, k, rounds = 16, 3, 30_000
    p_log = rng.normal(size=V) * 1.2
    q_log = p_log + rng.normal(size=V) * 1.0
    p = OV.softmax_at(p_log, 1.0)
    q = OV.softmax_at(q_log, 1.0)
    T = k + 1
    parent = np.tile(np.array([-1] + [0] * k), rounds)
    no = np.arange(rounds + 1) * T
    tgt = np.tile(p_log, (rounds * T, 1))
    drf = q_log[None, :]
    drow = np.zeros(rounds * T, dtype=np.int64)
    tokens = rng.choice(V, size=rounds * T, p=q)
    uni = rng.random((rounds * T, 2))
    res = OV.verify(tgt, drf, OV.DRAFT_LOGITS, drow, tokens, parent, no, uni, 1.0, V,
                    max_path=T, T_max=T)
    first = np.array([t[0] for t in res["out_tokens"]])
    counts = np.bincount(first, minlength=V)
    stat = chisquare(counts, p * rounds)
    assert stat.pvalue > 0.01, stat


def test_greedy_is_the_low_temperature_limit():
    rng = np.random.default_rng(3)
    V, gamma, B = 50, 5, 200
    T = gamma + 1
    tgt = rng.normal(size=(B * T, V)) * 3
    drf = tgt + rng.normal(size=(B * T, V)) * 0.7
    # keep cases where top-2 gaps are clear so tau = 1e-4 is numerically greedy
    tokens = np.zeros(B * T, dtype=np.int64)
    for r in range(B):
        for i in range(gamma):
            tokens[r * T + i + 1] = int(np.argmax(drf[r * T + i]))   # greedy drafts
    parent = np.tile(np.array([-1] + list(range(gamma))), B)
    no = np.arange(B + 1) * T
    uni = rng.random((B * T, 2))
    drow = np.arange(B * T)
    g = OV.verify(tgt, drf, OV.DRAFT_LOGITS, drow, tokens, parent, no, uni, 0.0, V, T, T_max=T)
    s = OV.verify(tgt, drf, OV.DRAFT_LOGITS, drow, tokens, parent, no, uni, 1e-4, V, T, T_max=T)
    srt = np.sort(np.concatenate([tgt, drf]), axis=1)
    clear = (srt[:, -1] - srt[:, -2]).reshape(2, B, T).min(axis=(0, 2)) > 0.02
    assert clear.sum() > B // 2
    for r in np.nonzero(clear)[0]:
        assert g["out_tokens"][r] == s["out_tokens"][r]
        assert g["path"][r] == s["path"][r]
    # every accepted greedy token is the target argmax along the path; the last is argmax too
    for r in range(B):
        path = g["path"][r]
        for d in range(len(path)):
            assert g["out_tokens"][r][d] == int(np.argmax(tgt[r * T + path[d]]))


def test_greedy_ties_go_to_lowest_token():
    V = 8
    tgt = np.zeros((2, V))
    tgt[0, [2, 5]] = 4.0
    tgt[1, [1, 6]] = 9.0
    res = OV.verify(tgt, np.zeros((1, V)), OV.DRAFT_LOGITS, [0, -1], [0, 2], [-1, 0], [0, 2],
                    np.zeros((2, 2)), 0.0, V, 2, T_max=2)
    assert res["out_tokens"][0] == [2, 1]


def test_inverse_cdf_and_its_distance_to_the_edges():
    """The smallest x with sum_{y <= x} w(y) > u * sum(w), and the distance from u to the nearer
    edge of x's CDF interval (what the parity tests read to exempt draws near an edge)."""
    w = [1.0, 2.0, 3.0, 4.0]                  # CDF edges 0, 0.1, 0.3, 0.6, 1
    for u, x, gap in ((0.0, 0, 0.0), (0.05, 0, 0.05), (0.25, 1, 0.05), (0.3, 2, 0.0),
                      (0.5, 2, 0.1), (0.61, 3, 0.01), (0.99, 3, 0.01)):
        got_x, got_gap = OV.inverse_cdf(w, u)
        assert got_x == x, u
        assert abs(got_gap - gap) < 1e-15, u


def test_recorded_ratios_are_p_over_q():
    """Every ("test", node, child, a, u) event carries a = p(tok) / q(tok) of the child's token
    (the first sibling's plain ratio), with p and q the library's softmax at tau."""
    from scipy.special import softmax
    rng = np.random.default_rng(21)
    V, T, tau = 30, 5, 0.8
    tgt = rng.normal(size=(T, V)) * 2
    drf = rng.normal(size=(T, V)) * 2
    tokens = [0] + [int(x) for x in rng.integers(0, V, T - 1)]
    uni = np.full((T, 2), 1e-9)                  # every test passes: the walk goes to the leaf
    res = OV.verify(tgt, drf, OV.DRAFT_LOGITS, np.arange(T), tokens, list(range(-1, T - 1)),
                    [0, T], uni, tau, V, T, T_max=T)
    tests = [e for e in res["events"][0] if e[0] == "test"]
    assert [e[2] for e in tests] == [1, 2, 3, 4]
    for _, node, c, a, u in tests:
        want = softmax(tgt[node] / tau)[tokens[c]] / softmax(drf[node] / tau)[tokens[c]]
        assert abs(a - want) < 1e-12 * want and u == 1e-9


def test_greedy_walk_on_a_hand_made_tree():
    """tau = 0 on a tree whose argmaxes are set by hand: the root's children 1, 2, 3 carry
    tokens 5, 6, 7 and the root's argmax is 6 (child 1 rejected, child 2 accepted); node 2's
    children 4, 5 carry tokens 1, 2 and its argmax is 2 (child 4 rejected, child 5 accepted);
    node 5 is a leaf, whose argmax 3 is the bonus token.  Two rejections in all."""
    V = 8
    parent = [-1, 0, 0, 0, 2, 2]
    tokens = [0, 5, 6, 7, 1, 2]
    tgt = np.zeros((6, V))
    tgt[0, 6] = tgt[2, 2] = tgt[5, 3] = 1.0
    res = OV.verify(tgt, np.zeros((6, V)), OV.DRAFT_LOGITS, np.arange(6), tokens, parent, [0, 6],
                    np.zeros((6, 2)), 0.0, V, 4, T_max=6)
    assert res["path"][0] == [0, 2, 5]
    assert res["out_tokens"][0] == [6, 2, 3]
    assert res["rejections"][0] == 2 and res["n_acc"][0] == 2 and res["out_len"][0] == 3


def test_a_draft_token_with_zero_draft_probability():
    """min(1, p / q) with q(x) = 0: p / q is +inf when p(x) > 0 (accepted whatever u is) and the
    test fails when p(x) = 0 as well (rejected whatever u is)."""
    V = 4
    q = np.array([[0.5, 0.5, 0.0, 0.0]])
    tgt = np.zeros((2, V))
    tgt[0, 3] = -1e4                     # p(3) = 0 in fp64
    for tok, accepted in ((2, True), (3, False)):
        for u in (0.0, 0.999999):
            res = OV.verify(tgt, q, OV.DRAFT_PROBS, [0, 0], [0, tok], [-1, 0], [0, 2],
                            np.array([[0.5, 0.5], [u, 0.5]]), 1.0, V, 2, T_max=2)
            assert (res["n_acc"][0] == 1) == accepted, (tok, u)


def test_data_errors_flagged():
    V = 10
    tgt = np.zeros((3, V))
    base = dict(target=tgt, draft=np.zeros((2, V)), draft_kind=OV.DRAFT_LOGITS,
                parent=[-1, 0, 1], node_offset=[0, 3], uniforms=np.zeros((3, 2)), tau=1.0, V=V)
    r = OV.verify(draft_row=[0, 1, -1], tokens=[0, 3, V], max_path=3, **base)
    assert r["status"][0] == OV.BAD_TOKEN and r["out_len"][0] == 0 and r["n_acc"][0] == -1
    r = OV.verify(draft_row=[0, 2, -1], tokens=[0, 3, 4], max_path=3, **base)
    assert r["status"][0] == OV.BAD_DRAFT_ROW
    r = OV.verify(draft_row=[0, 1, -1], tokens=[0, 3, 4], max_path=2, **base)
    assert r["status"][0] == OV.BAD_DEPTH
    r = OV.verify(draft_row=[0, 1, -1], tokens=[0, 3, 4], max_path=3, **base)
    assert r["status"][0] == 0 and r["out_len"][0] >= 1
    # greedy reads no draft row: an out-of-range one is not an error at tau = 0
    r = OV.verify(draft_row=[-1, 9, -1], tokens=[0, 3, 4], max_path=3,
                  **dict(base, tau=0.0))
    assert r["status"][0] == 0 and r["out_len"][0] >= 1
    # multi-draft: each drafted node names the row it was drawn from; the rows its parent
    # would name are not read
    multi = dict(base, sibling_rule=OV.SIBLING_MULTI_DRAFT)
    r = OV.verify(draft_row=[-1, 0, 1], tokens=[0, 3, 4], max_path=3, **multi)
    assert r["status"][0] == 0
    r = OV.verify(draft_row=[0, 1, 2], tokens=[0, 3, 4], max_path=3, **multi)
    assert r["status"][0] == OV.BAD_DRAFT_ROW


@pytest.mark.parametrize("rule", [OV.SIBLING_RESIDUAL, OV.SIBLING_MULTI_DRAFT])
def test_zero_residual_mass_draws_from_p(rule):
    """Draft probabilities q = 2p (not normalised, as a caller may pass them): the test
    accepts with p / q = 1/2, and after a rejection max(0, p - q) is 0 everywhere, so the final
    token is drawn from p itself, by the inverse CDF over ascending token id."""
    V = 5
    logits = np.array([0.3, -1.0, 1.2, 0.0, 0.7])
    p = np.exp(logits - logits.max())
    p /= p.sum()
    q = 2.0 * p
    for u_samp in (0.05, 0.4, 0.75, 0.97):
        uni = np.array([[0.5, u_samp], [0.6, 0.5]])   # u_acc = 0.6 >= 1/2: rejected
        res = OV.verify(np.stack([logits, logits]), q[None, :], OV.DRAFT_PROBS, [0, 0], [0, 2],
                        [-1, 0], [0, 2], uni, 1.0, V, 2, sibling_rule=rule, T_max=2)
        want = int(np.nonzero(np.cumsum(p) > u_samp)[0][0])
        assert res["path"][0] == [0] and res["rejections"][0] == 1
        assert res["out_tokens"][0] == [want], (u_samp, res["out_tokens"][0], want)
