"""Oracle: ratio-test verification of a draft tree, fp64.

Follows:
  * "推测解码 2026" (guijiagi.com), 数学基础：拒绝采样: accept a drafted token x with probability
    min(1, p(x)/q(x)) (always when p >= q); on rejection resample from the adjusted
    distribution relu(p - q), normalised, and drop every later candidate;
  * "【模型后训练与深度推理】9 推理加速：推测解码与级联推理" (kapook.pages.dev / CSDN), section 7.1: the
    acceptance probability alpha_i = min(1, p/q) and the residual norm(max(0, p - q)), with the
    output distribution equal to p; section 7.2: the emitted count L includes the final
    corrected (or bonus) token;
  * "投机推理算法的常见优化手段" (cnblogs zrq96), 草稿树的验证——树形掩码: the logits at tree node i give
    P(. | ancestors(i)), and tree verification walks every level of the tree instead of one
    sequence;
  * "万字综述 10+ 种 LLM 投机采样推理加速方案" (m.haoling.cc), section 4.3: argmax sampling (temp = 0)
    as the greedy special case.

Readings where the pages are silent (each one is listed in the design notes):
  * the children of node i are tested in increasing node index against q_i, the draft
    distribution i's children were proposed from (draft_row[i]);
  * siblings (SIBLING_RESIDUAL, default): after k rejections at node i the target is the k-fold
    residual, which in closed form is R_k = max(0, p - C_k q) with C_0 = 0, N_k = sum R_k,
    C_{k+1} = C_k + N_k (because max(0, max(0, p - a q) - b q) = max(0, p - (a + b) q) for
    a, b >= 0); child k is accepted iff u_acc < R_k(tok) / (N_k q(tok)), which for k = 0 is
    exactly p/q.  SIBLING_INDEPENDENT tests every sibling with p/q and resamples from
    max(0, p - q);
  * SIBLING_MULTI_DRAFT (several draft models proposing siblings: "万字综述 10+ 种 LLM 投机采样推理
    加速方案" 5.1, a group of small models predicting together; "投机推理算法的常见优化手段" 草稿树的生成,
    merge-based trees built from k small models): draft_row[c] is the row child c itself was
    drawn from, so siblings carry their own q_c.  The pages' rule is applied sibling after
    sibling with no closed form: the running target starts as r = p, child c is accepted iff
    u_acc < r(tok) / q_c(tok), and a rejection replaces r by norm(max(0, r - q_c));
  * a zero residual mass (N_k = 0: through rounding for normalised rows, exactly for draft
    probabilities that sum to more than 1, e.g. q = 2p) stops the sibling loop and the final
    token is drawn from p;
  * tau applies to target and draft logits alike; draft probabilities are used as given;
    tau = 0 accepts a child iff its token is argmax p_i (lowest id on ties) and the final token
    is argmax p at the stop node;
  * inverse CDF over ascending token id: the smallest x with sum_{y<=x} w(y) > u * sum_y w(y);
  * a leaf at the end of a fully accepted path yields a bonus token drawn from p_leaf.
"""
import numpy as np

from .tree import tree_build

SIBLING_RESIDUAL = 0
SIBLING_INDEPENDENT = 1
SIBLING_MULTI_DRAFT = 2
DRAFT_LOGITS = 0
DRAFT_PROBS = 1

BAD_TOKEN = 4
BAD_DRAFT_ROW = 8
BAD_DEPTH = 16


def softmax_at(x, tau):
    """p = softmax(x / tau), fp64."""
    y = np.asarray(x, dtype=np.float64) / tau
    e = np.exp(y - y.max())
    return e / e.sum()


def draft_q(draft, drow, V, tau, draft_kind):
    """q of draft row drow: softmax(row / tau) for draft logits, the row itself for draft
    probabilities."""
    row = draft[drow, :V]
    return softmax_at(row, tau) if draft_kind == DRAFT_LOGITS else np.asarray(row, np.float64)


def inverse_cdf(w, u):
    """Smallest x with cumsum(w)[x] > u * sum(w).  Returns (x, gap) where gap is the distance,
    in units of u, from u to the nearer edge of x's CDF interval."""
    c = np.cumsum(np.asarray(w, dtype=np.float64))
    total = c[-1]
    x = int(np.searchsorted(c, u * total, side="right"))
    x = min(x, len(c) - 1)
    lo = c[x - 1] / total if x > 0 else 0.0
    hi = c[x] / total
    return x, min(u - lo, hi - u)


def verify(target, draft, draft_kind, draft_row, tokens, parent, node_offset, uniforms, tau,
           V, max_path, sibling_rule=SIBLING_RESIDUAL, T_max=256):
    """Verify every request of a packed batch of draft trees.

    target: [N, >=V] target logits (row n = next-token logits at node n); draft: [R, >=V] draft
    logits or probabilities; draft_row: [N]; tokens: [N]; parent: [N] local; node_offset: [B+1];
    uniforms: [N, 2] = (u_acc, u_samp).

    Returns dict(status[B], n_acc[B] (-1 for a bad request), path[B] (lists of local node ids,
    root first), out_tokens[B] (accepted draft tokens then the final token), out_len[B],
    rejections[B], final_kind[B] ("bonus" | "correction" | None), events[B]).  events lists the
    comparisons taken: ("test", node, child, a, u) and ("sample", node, u, gap).
    """
    target = np.asarray(target)
    draft = np.asarray(draft)
    draft_row = np.asarray(draft_row, dtype=np.int64)
    tokens = np.asarray(tokens, dtype=np.int64)
    uniforms = np.asarray(uniforms, dtype=np.float64)
    node_offset = np.asarray(node_offset, dtype=np.int64)
    B = len(node_offset) - 1
    R = draft.shape[0]
    tb = tree_build(parent, node_offset, np.zeros(B, dtype=np.int64), T_max)
    status = tb["status"].copy()
    res = dict(status=status, n_acc=np.full(B, -1, dtype=np.int64), path=[[] for _ in range(B)],
               out_tokens=[[] for _ in range(B)], out_len=np.zeros(B, dtype=np.int64),
               rejections=np.zeros(B, dtype=np.int64), final_kind=[None] * B,
               events=[[] for _ in range(B)])
    for r in range(B):
        o, T = int(node_offset[r]), int(node_offset[r + 1] - node_offset[r])
        if status[r]:
            continue
        par = np.asarray(parent[o:o + T], dtype=np.int64)
        kids_of = [[c for c in range(T) if par[c] == i] for i in range(T)]
        if any(not (0 <= tokens[o + c] < V) for c in range(1, T)):
            status[r] |= BAD_TOKEN
        if sibling_rule == SIBLING_MULTI_DRAFT:
            # every drafted node names the row it was drawn from
            if tau > 0 and any(not (0 <= draft_row[o + c] < R) for c in range(1, T)):
                status[r] |= BAD_DRAFT_ROW
        elif tau > 0 and any(kids_of[i] and not (0 <= draft_row[o + i] < R) for i in range(T)):
            status[r] |= BAD_DRAFT_ROW
        if int(tb["depth"][o:o + T].max()) + 1 > max_path:
            status[r] |= BAD_DEPTH
        if status[r]:
            continue
        node, path, events, rejections = 0, [0], [], 0
        while True:
            kids = kids_of[node]
            if tau == 0:
                best = int(np.argmax(np.asarray(target[o + node, :V], dtype=np.float64)))
                nxt = None
                for c in kids:
                    if tokens[o + c] == best:
                        nxt = c
                        break
                    rejections += 1
                if nxt is None:
                    final, kind = best, ("bonus" if not kids else "correction")
                    break
                path.append(nxt)
                node = nxt
                continue
            p = softmax_at(target[o + node, :V], tau)
            u_samp = float(uniforms[o + node, 1])
            if not kids:
                final, gap = inverse_cdf(p, u_samp)
                events.append(("sample", node, u_samp, gap))
                kind = "bonus"
                break
            def q_of(drow):
                return draft_q(draft, drow, V, tau, draft_kind)

            if sibling_rule == SIBLING_MULTI_DRAFT:
                target_now, accepted, w_final = p, None, None
                for c in kids:
                    tok = int(tokens[o + c])
                    qc = q_of(draft_row[o + c])
                    num, den = target_now[tok], qc[tok]
                    a = num / den if den > 0 else (np.inf if num > 0 else 0.0)
                    u = float(uniforms[o + c, 0])
                    events.append(("test", node, c, a, u))
                    if u < a:
                        accepted = c
                        break
                    rejections += 1
                    resid = np.maximum(0.0, target_now - qc)
                    mass = resid.sum()
                    if mass <= 0.0:
                        w_final = p
                        break
                    target_now = resid / mass
                if accepted is not None:
                    path.append(accepted)
                    node = accepted
                    continue
                final, gap = inverse_cdf(target_now if w_final is None else w_final, u_samp)
                events.append(("sample", node, u_samp, gap))
                kind = "correction"
                break
            q = q_of(draft_row[o + node])
            C, Nk = 0.0, 1.0
            accepted, w_final = None, None
            for c in kids:
                tok = int(tokens[o + c])
                if sibling_rule == SIBLING_RESIDUAL:
                    Rk = p if C == 0.0 else np.maximum(0.0, p - C * q)
                    num, den = Rk[tok], Nk * q[tok]
                else:
                    num, den = p[tok], q[tok]
                a = num / den if den > 0 else (np.inf if num > 0 else 0.0)
                u = float(uniforms[o + c, 0])
                events.append(("test", node, c, a, u))
                if u < a:
                    accepted = c
                    break
                rejections += 1
                if sibling_rule == SIBLING_RESIDUAL:
                    C = C + Nk
                    Nk = np.maximum(0.0, p - C * q).sum()
                    if Nk <= 0.0:
                        w_final = p
                        break
            if accepted is not None:
                path.append(accepted)
                node = accepted
                continue
            if w_final is None:
                w_final = np.maximum(0.0, p - (C if sibling_rule == SIBLING_RESIDUAL else 1.0) * q)
                if w_final.sum() <= 0.0:
                    w_final = p
            final, gap = inverse_cdf(w_final, u_samp)
            events.append(("sample", node, u_samp, gap))
            kind = "correction"
            break
        res["n_acc"][r] = len(path) - 1
        res["path"][r] = path
        res["out_tokens"][r] = [int(tokens[o + c]) for c in path[1:]] + [int(final)]
        res["out_len"][r] = len(path)
        res["rejections"][r] = rejections
        res["final_kind"][r] = kind
        res["events"][r] = events
    return res
