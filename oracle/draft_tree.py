"""Oracle: building the draft tree on the device -- EAGLE-2's expansion of the most probable
leaves and ECHO's batch-wide budget -- the step before verification.

Follows "投机推理算法的常见优化手段" (cnblogs zrq96): section 草稿树的生成 -- an expansion-based tree
takes the top-K tokens at every drafting step; EAGLE-2 expands, at each step, only the K most
probable leaves of the newest level, ranking a leaf by the product of the probabilities along
its path (equivalently, it extends only the most probable paths); section 动态草稿长度 -- ECHO fixes
a global budget K_max of tokens verified per step, shared by every request of the batch, so
confident requests get deeper or wider trees and others give theirs up.

Readings (the page names the quantities, not the procedure's details):
  * a candidate's score is the sum of draft log-probabilities along its path,
    log q(child) = log_softmax(draft_row / tau)[token], the root's score is 0;
  * the top-K tokens of a row are ordered by log-probability, ties to the lower token id;
  * level 1 expands the root; level l > 1 expands the K best candidates of level l - 1 of each
    request (ties to the lower candidate index); expanded candidates are taken in increasing
    candidate index, and the children of one are appended in top-K order;
  * ECHO keeps every root and the K_max - B best non-root candidates of the batch (ties by
    request, then candidate index); a child's score never exceeds its parent's (log q <= 0), so
    the kept set is closed under ancestors;
  * the packed tree keeps each request's kept candidates in candidate-index order (parents
    first); a node's draft row is the row its expansion produced if one of its children was
    kept, else -1.
Everything is fp64.
"""
import numpy as np


def log_softmax(row, tau=1.0):
    """fp64 log_softmax(row / tau), by the definition (shifted by the row maximum)."""
    y = np.asarray(row, dtype=np.float64) / tau
    m = y.max()
    return y - (m + np.log(np.exp(y - m).sum()))


def topk(row, k, tau=1.0):
    """The k tokens with the largest log-probability (ties to the lower id), best first, and
    their log-probabilities.  Every token at or above the k-th largest value is a candidate
    (a library partition finds that value); the candidates are ordered by (value descending,
    id) and the first k kept."""
    lq = log_softmax(row, tau)
    n = len(lq)
    k = min(k, n)
    kth = np.partition(lq, n - k)[n - k]
    cand = np.nonzero(lq >= kth)[0]
    order = sorted(cand.tolist(), key=lambda x: (-lq[x], x))[:k]
    return np.array(order, dtype=np.int64), lq[order]


class Pool:
    """Per request: the candidates made so far -- parent (candidate index), token, depth,
    score and the draft row produced when the candidate was expanded (-1 if never)."""

    def __init__(self, roots):
        self.cands = [[dict(parent=-1, token=int(t), depth=0, score=0.0, row=-1)] for t in roots]

    @property
    def B(self):
        return len(self.cands)


def expand_select(pool, level, K):
    """Which candidates to expand at `level`: the root at level 1, else the K best (score, then
    lower index) of depth level - 1.  Returns per request the chosen candidate indices in
    increasing order."""
    out = []
    for r, cs in enumerate(pool.cands):
        if level == 1:
            out.append([0])
            continue
        front = [i for i, c in enumerate(cs) if c["depth"] == level - 1]
        best = sorted(front, key=lambda i: (-cs[i]["score"], i))[:K]
        out.append(sorted(best))
    return out


def append_children(pool, chosen, row_ids, tops, level):
    """chosen[r] = expanded candidate indices (increasing); row_ids[r][j] = the draft row of the
    j-th; tops[r][j] = (tokens, logps) of that row's top-K.  Appends the children in order."""
    for r, cs in enumerate(pool.cands):
        for j, i in enumerate(chosen[r]):
            cs[i]["row"] = int(row_ids[r][j])
            toks, lps = tops[r][j]
            for t, lp in zip(toks, lps):
                cs.append(dict(parent=i, token=int(t), depth=level, score=cs[i]["score"] + float(lp),
                               row=-1))


def echo_select(pool, K_max):
    """Kept candidate indices per request: every root plus the K_max - B best non-root
    candidates of the batch (score, then request, then index)."""
    nonroot = [(r, i) for r, cs in enumerate(pool.cands) for i in range(1, len(cs))]
    nonroot.sort(key=lambda ri: (-pool.cands[ri[0]][ri[1]]["score"], ri[0], ri[1]))
    keep = set((r, 0) for r in range(pool.B)) | set(nonroot[:max(0, K_max - pool.B)])
    return [sorted(i for i in range(len(cs)) if (r, i) in keep) for r, cs in enumerate(pool.cands)]


def pack(pool, kept):
    """The verification layout of the kept candidates: node_offset [B+1], parent [N] (local,
    -1 for roots), tokens [N], depth [N], draft_row [N] and source (request, candidate) [N]."""
    node_offset, parent, tokens, depth, draft_row, source = [0], [], [], [], [], []
    for r, cs in enumerate(pool.cands):
        local = {old: new for new, old in enumerate(kept[r])}
        has_kept_child = set(cs[i]["parent"] for i in kept[r] if i > 0)
        for old in kept[r]:
            c = cs[old]
            parent.append(-1 if c["parent"] < 0 else local[c["parent"]])
            tokens.append(c["token"])
            depth.append(c["depth"])
            draft_row.append(c["row"] if old in has_kept_child else -1)
            source.append((r, old))
        node_offset.append(node_offset[-1] + len(kept[r]))
    as_i = lambda x: np.asarray(x, dtype=np.int64)
    return dict(node_offset=as_i(node_offset), parent=as_i(parent), tokens=as_i(tokens),
                depth=as_i(depth), draft_row=as_i(draft_row), source=source)


def build(roots, rows_of_level, K, depth, K_max, tau=1.0):
    """The whole construction: rows_of_level(level, chosen) returns, for the candidates chosen
    at that level, (row_ids[r][j], rows[r][j]) -- the draft model's output, an input here.
    Returns (pool, kept, packed)."""
    pool = Pool(roots)
    for level in range(1, depth + 1):
        chosen = expand_select(pool, level, K)
        if not any(chosen):
            break
        row_ids, rows = rows_of_level(level, chosen)
        tops = [[topk(rows[r][j], K, tau) for j in range(len(chosen[r]))] for r in range(pool.B)]
        append_children(pool, chosen, row_ids, tops, level)
    kept = echo_select(pool, K_max)
    return pool, kept, pack(pool, kept)
