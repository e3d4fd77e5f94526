"""Pins for oracle.lookahead: the lookahead-decoding mask.

  * a hand-derived worked example (tests/golden/lookahead_w3_n3_g2.txt);
  * the page's counts: W x (N - 1) lookahead tokens (with "0"), G x (N - 1) verify tokens, and
    the per-step compute multiple W(N-1) + G(N-1) ((W, N, G) = (5, 4, 5) -> 30, and the 120 /
    80 / 56 the page quotes for 7B / 13B / 33B models, read as G = W, N = 5);
  * rule 1 (causal) and rule 2 (branches mutually invisible) checked on every pair;
  * N = 2 is Jacobi decoding: one causal sequence of W tokens;
  * every token sees one token per position 0 .. its own (a consistent causal sequence), so
    each collected n-gram is one;
  * the mask is an ancestor mask: the tree build of the derived parent array reproduces it, with
    depth = position.
"""
import os

import numpy as np
import pytest

from oracle import lookahead as OL
from oracle import tree as OT

GOLD = os.path.join(os.path.dirname(__file__), "golden", "lookahead_w3_n3_g2.txt")


def _golden():
    par = pos = None
    rows = []
    with open(GOLD, encoding="utf-8") as f:
        lines = f.read().splitlines()
    for line in lines:
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        if f[0] == "parent":
            par = [int(x) for x in f[1:]]
        elif f[0] == "position":
            pos = [int(x) for x in f[1:]]
        else:
            rows.append([int(x) for x in f[1:]])
    return par, pos, np.asarray(rows, dtype=bool)


def test_worked_example():
    par, pos, mask = _golden()
    np.testing.assert_array_equal(OL.lookahead_mask(3, 3, 2), mask)
    assert OL.lookahead_parents(3, 3, 2).tolist() == par
    assert [OL.position(n) for n in OL.lookahead_nodes(3, 3, 2)] == pos


@pytest.mark.parametrize("W,N,G,mult", [(5, 4, 5, 30), (15, 5, 15, 120), (10, 5, 10, 80),
                                        (7, 5, 7, 56)])
def test_counts(W, N, G, mult):
    nodes = OL.lookahead_nodes(W, N, G)
    look = [n for n in nodes if n[0] != "verify"]
    ver = [n for n in nodes if n[0] == "verify"]
    assert len(look) == W * (N - 1)
    assert len(ver) == G * (N - 1)
    assert len(nodes) == mult


@pytest.mark.parametrize("W,N,G", [(5, 4, 5), (4, 2, 3), (6, 6, 2), (1, 3, 0), (7, 5, 7)])
def test_rules(W, N, G):
    nodes = OL.lookahead_nodes(W, N, G)
    m = OL.lookahead_mask(W, N, G)
    for i, a in enumerate(nodes):
        assert m[i, i] and m[i, 0]
        for j, b in enumerate(nodes):
            if m[i, j] and i != j:
                assert OL.position(b) < OL.position(a)                 # rule 1
            if {a[0], b[0]} == {"look", "verify"}:
                assert not m[i, j]                                      # rule 2
        # one visible token per position 0 .. own position
        seen = sorted(OL.position(nodes[j]) for j in np.flatnonzero(m[i]))
        assert seen == list(range(OL.position(a) + 1))


def test_n2_is_jacobi_decoding():
    m = OL.lookahead_mask(6, 2, 0)
    np.testing.assert_array_equal(m, np.tril(np.ones((6, 6), dtype=bool)))


@pytest.mark.parametrize("W,N,G", [(5, 4, 5), (15, 5, 15), (3, 6, 4)])
def test_is_an_ancestor_mask(W, N, G):
    par = OL.lookahead_parents(W, N, G)
    T = len(par)
    assert par[0] == -1 and all(0 <= par[i] < i for i in range(1, T))
    tb = OT.tree_build(par, [0, T], [100], T)
    assert not tb["status"].any()
    np.testing.assert_array_equal(tb["mask"][0], OL.lookahead_mask(W, N, G))
    assert tb["pos_id"].tolist() == [100 + OL.position(n) for n in OL.lookahead_nodes(W, N, G)]


def test_diagonals_are_the_collected_ngrams():
    # the n-gram through step 0 at position p0 is (0, p0), (1, p0+1), ..., (N-2, p0+N-2): each
    # token on it sees the previous one
    W, N = 5, 4
    nodes = OL.lookahead_nodes(W, N, 0)
    idx = {n: i for i, n in enumerate(nodes)}
    m = OL.lookahead_mask(W, N, 0)
    for p0 in range(1, W):
        diag = [("look", l, p0 + l) for l in range(N - 1)]
        for a, b in zip(diag[1:], diag[:-1]):
            assert m[idx[a], idx[b]]
