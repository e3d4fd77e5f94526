"""Pins for oracle.draft_tree (EAGLE-2 expansion of the most probable leaves + ECHO's batch-wide
budget, "投机推理算法的常见优化手段" 草稿树的生成 and 动态草稿长度).

  * log_softmax against scipy's; top-K against a brute-force sort of a hand-made row with ties;
  * the page's counts: with K = 5, level 2 holds 25 leaves and level 3 expands only 5 of them;
    with every candidate kept a depth-8 tree holds 1 + 5 + 7 * 25 = 181 tokens;
  * "expand the most probable paths": the expanded leaves are the K largest PRODUCTS of the draft
    probabilities along the path, recomputed here by multiplying softmax values;
  * ECHO: exactly K_max tokens kept over the batch, every root kept, every kept non-root at
    least as probable as every dropped one, the kept set closed under ancestors; a request with
    confident (peaked) draft rows ends up with a larger and deeper tree than a flat one;
  * the packed layout is a valid tree (the tree build accepts it, depths agree).
"""
import numpy as np
import pytest
from scipy.special import log_softmax as sp_log_softmax
from scipy.special import softmax as sp_softmax

from oracle import draft_tree as OD
from oracle import tree as OT


def test_log_softmax_and_topk():
    rng = np.random.default_rng(0)
    for tau in (1.0, 0.5, 2.0):
        x = rng.normal(size=50) * 3
        np.testing.assert_allclose(OD.log_softmax(x, tau), sp_log_softmax(x / tau), atol=1e-12)
    row = np.array([1.0, 3.0, 3.0, 2.0, 3.0, -1.0])
    toks, lps = OD.topk(row, 2)
    assert toks.tolist() == [1, 2]
    toks, lps = OD.topk(row, 5)
    assert toks.tolist() == [1, 2, 4, 3, 0]
    np.testing.assert_allclose(lps, sp_log_softmax(row)[[1, 2, 4, 3, 0]], atol=1e-12)
    toks, lps = OD.topk(row, 10)             # K above the vocabulary: every token, best first
    assert toks.tolist() == [1, 2, 4, 3, 0, 5]


def _random_build(B, V, K, D, K_max, seed, peaked=(), tau=1.0):
    rng = np.random.default_rng(seed)
    store = {}

    def rows_of_level(level, chosen):
        row_ids, rows = [], []
        for r in range(len(chosen)):
            ids, rr = [], []
            for j, i in enumerate(chosen[r]):
                scale = 8.0 if r in peaked else 0.3
                row = rng.normal(size=V) * scale
                rid = len(store)
                store[rid] = row
                ids.append(rid)
                rr.append(row)
            row_ids.append(ids)
            rows.append(rr)
        return row_ids, rows

    roots = rng.integers(0, V, size=B)
    pool, kept, packed = OD.build(roots, rows_of_level, K, D, K_max, tau)
    return pool, kept, packed, store


def test_counts_of_the_page():
    pool, kept, packed, _ = _random_build(B=2, V=30, K=5, D=8, K_max=10 ** 6, seed=1)
    for cs in pool.cands:
        per_depth = np.bincount([c["depth"] for c in cs])
        assert per_depth.tolist() == [1, 5] + [25] * 7
        assert len(cs) == 181
        expanded_at = np.bincount([c["depth"] for c in cs if c["row"] >= 0], minlength=9)
        assert expanded_at.tolist() == [1] + [5] * 7 + [0]
    assert packed["node_offset"].tolist() == [0, 181, 362]


def test_expanded_leaves_are_the_most_probable_paths():
    pool, kept, packed, store = _random_build(B=3, V=12, K=3, D=4, K_max=10 ** 6, seed=2)
    for cs in pool.cands:
        def path_prob(i):   # product of the draft probabilities along the path
            pr = 1.0
            while cs[i]["parent"] >= 0:
                p = cs[i]["parent"]
                pr *= sp_softmax(store[cs[p]["row"]])[cs[i]["token"]]
                i = p
            return pr
        for level in range(1, 4):
            front = [i for i, c in enumerate(cs) if c["depth"] == level]
            chosen = [i for i in front if cs[i]["row"] >= 0]
            if level < 4:
                assert len(chosen) == min(3, len(front))
            probs = {i: path_prob(i) for i in front}
            worst_chosen = min(probs[i] for i in chosen)
            assert all(probs[i] <= worst_chosen * (1 + 1e-12) for i in front if i not in chosen)


@pytest.mark.parametrize("K_max", [8, 40, 100])
def test_echo_budget(K_max):
    pool, kept, packed, _ = _random_build(B=4, V=20, K=3, D=5, K_max=K_max, seed=3)
    total = sum(len(k) for k in kept)
    assert total == min(K_max, sum(len(cs) for cs in pool.cands))
    for r, cs in enumerate(pool.cands):
        assert kept[r][0] == 0
        ks = set(kept[r])
        for i in kept[r]:
            if i > 0:
                assert cs[i]["parent"] in ks          # closed under ancestors
    kept_scores = [pool.cands[r][i]["score"] for r in range(4) for i in kept[r] if i > 0]
    dropped = [c["score"] for r, cs in enumerate(pool.cands) for i, c in enumerate(cs)
               if i > 0 and i not in kept[r]]
    if kept_scores and dropped:
        assert min(kept_scores) >= max(dropped)


def test_confident_requests_get_the_budget():
    pool, kept, packed, _ = _random_build(B=2, V=40, K=4, D=6, K_max=40, seed=4, peaked=(0,))
    sizes = [len(k) for k in kept]
    depths = [max(pool.cands[r][i]["depth"] for i in kept[r]) for r in range(2)]
    assert sizes[0] > sizes[1] and depths[0] > depths[1]


@pytest.mark.parametrize("tau", [1.0, 0.5])
def test_scores_are_path_log_probabilities(tau):
    """Every score is the sum of scipy's log_softmax(row / tau)[token] along the path (the
    root's is 0), and an expanded candidate's children are its row's K most probable tokens at
    that temperature, best first."""
    pool, kept, packed, store = _random_build(B=2, V=15, K=3, D=3, K_max=10 ** 6, seed=6, tau=tau)
    for cs in pool.cands:
        assert cs[0]["score"] == 0.0
        for c in cs[1:]:
            lp = sp_log_softmax(store[cs[c["parent"]]["row"]] / tau)
            assert abs(c["score"] - (cs[c["parent"]]["score"] + lp[c["token"]])) < 1e-12
        for i, c in enumerate(cs):
            if c["row"] >= 0:
                lp = sp_log_softmax(store[c["row"]] / tau)
                kids = [x["token"] for x in cs if x["parent"] == i]
                assert kids == np.argsort(-lp, kind="stable")[:3].tolist()


def test_echo_ties_go_to_the_lower_request_then_the_lower_candidate():
    # both requests draft from the same row, whose two best tokens tie: all four non-root
    # candidates have the same score
    row = np.array([2.0, 2.0, 1.0, 0.0, -1.0])

    def rows_of_level(level, chosen):
        return ([[0] * len(chosen[r]) for r in range(2)],
                [[row] * len(chosen[r]) for r in range(2)])

    for K_max, want in ((3, [[0, 1], [0]]), (4, [[0, 1, 2], [0]]), (5, [[0, 1, 2], [0, 1]])):
        pool, kept, packed = OD.build([7, 7], rows_of_level, 2, 1, K_max)
        assert [c["token"] for c in pool.cands[0][1:]] == [0, 1]
        assert kept == want, K_max


def test_packed_layout_is_a_tree():
    pool, kept, packed, _ = _random_build(B=5, V=25, K=3, D=4, K_max=37, seed=5)
    no = packed["node_offset"]
    T_max = int(np.diff(no).max())
    tb = OT.tree_build(packed["parent"], no, np.zeros(5, dtype=np.int64), T_max)
    assert not tb["status"].any()
    np.testing.assert_array_equal(tb["depth"], packed["depth"])
    for n, (r, old) in enumerate(packed["source"]):
        c = pool.cands[r][old]
        assert packed["tokens"][n] == c["token"]
        # a draft row only where a child was kept
        kept_children = [i for i in kept[r] if i > 0 and pool.cands[r][i]["parent"] == old]
        assert (packed["draft_row"][n] >= 0) == bool(kept_children)
        if kept_children:
            assert packed["draft_row"][n] == c["row"]
