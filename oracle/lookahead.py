"""Oracle: the lookahead-decoding attention mask (lookahead and verify branches in one forward),
written from the page's two rules and counts.

Follows "万字综述 10+ 种 LLM 投机采样推理加速方案" (m.haoling.cc), section 8 (前向解码 / Lookahead
Decoding): 8.2.1 -- a 2-D window of W future positions and N - 1 Jacobi steps, from which an
N-gram is collected along a diagonal (step 0 at position p, step 1 at p + 1, ..., plus the new
token); N = 2 is plain Jacobi decoding; 8.2.2 -- a verify branch of at most G candidate n-grams
whose first token matches the current token "0"; 8.2.3 -- both branches go into one forward
through a mask with two rules: (1) a token sees only tokens before it (causal), (2) lookahead
tokens and verify tokens do not see each other; the lookahead branch holds W x (N - 1) tokens
counting "0", the verify branch G x (N - 1).

Readings (the page draws the window but does not list its cells):
  * the window's step 0 holds "0" at position 0 and W - 1 tokens at positions 1 .. W - 1; step
    l = 1 .. N - 2 holds W tokens at positions l .. l + W - 1 (each step one position further
    ahead), so the branch has W (N - 1) tokens with "0", as the page counts;
  * "before it" for a lookahead token (l, p) is the Jacobi sequence its diagonal came from:
    the step-0 tokens at positions before the diagonal's start p - l, then the diagonal
    (0, p - l), (1, p - l + 1), ..., (l, p) -- so that a collected n-gram is a consistent
    causal sequence;
  * a verify candidate g is the chain "0", v(g, 1), ..., v(g, N - 1); it sees only its own
    earlier tokens and "0" (candidates are alternatives, not one sequence);
  * a token's position is its offset from "0" (p for (l, p), k for v(g, k)).
The node order is "0", step 0 by position, step 1 by position, ..., then each verify chain.
"""
import numpy as np


def lookahead_nodes(W, N, G):
    """The tokens in node order, as tuples: ("root",), ("look", l, p), ("verify", g, k)."""
    if W < 1 or N < 2 or G < 0:
        raise ValueError("need W >= 1, N >= 2, G >= 0")
    nodes = [("root",)]
    nodes += [("look", 0, p) for p in range(1, W)]
    for l in range(1, N - 1):
        nodes += [("look", l, p) for p in range(l, l + W)]
    for g in range(G):
        nodes += [("verify", g, k) for k in range(1, N)]
    return nodes


def position(node):
    if node[0] == "root":
        return 0
    return node[2]


def sees(a, b):
    """Does token a attend to token b (both from lookahead_nodes)?  The page's two rules with
    the readings above, written out case by case."""
    if a == b or b[0] == "root":
        return True
    if a[0] == "root":
        return False
    if a[0] != b[0]:
        return False                      # rule 2: the branches do not see each other
    if a[0] == "verify":
        _, ga, ka = a
        _, gb, kb = b
        return ga == gb and kb < ka       # own candidate, earlier tokens (rule 1)
    _, la, pa = a
    _, lb, pb = b
    start = pa - la                       # where a's diagonal leaves step 0
    if lb == 0 and 1 <= pb < start:
        return True                       # step-0 tokens before the diagonal (rule 1)
    return lb < la and pb - lb == start   # earlier tokens of a's own diagonal


def lookahead_mask(W, N, G):
    """Dense boolean mask [T, T]: mask[i, j] = token i attends to token j."""
    nodes = lookahead_nodes(W, N, G)
    T = len(nodes)
    m = np.zeros((T, T), dtype=bool)
    for i, a in enumerate(nodes):
        for j, b in enumerate(nodes):
            m[i, j] = sees(a, b)
    return m


def lookahead_parents(W, N, G):
    """The same structure as a parent array (every token sees exactly its ancestors): a token's
    parent is the latest token it sees other than itself."""
    nodes = lookahead_nodes(W, N, G)
    m = lookahead_mask(W, N, G)
    par = []
    for i, a in enumerate(nodes):
        seen = [j for j in range(len(nodes)) if m[i, j] and j != i]
        par.append(max(seen, key=lambda j: position(nodes[j])) if seen else -1)
    return np.asarray(par, dtype=np.int64)
