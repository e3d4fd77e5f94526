"""Oracle: tree attention over a paged KV cache, dense softmax in fp64.

Follows "投机推理算法的常见优化手段" (cnblogs zrq96), section 草稿树的验证——树形掩码: one forward
over the flattened tree with the ancestor mask, position ids and the KV cache, so that node i's
output is conditioned on its ancestors only; and "万字综述 10+ 种 LLM 投机采样推理加速方案"
(m.haoling.cc) section 5.2: tree-based parallel decoding shares the prefix through the mask
instead of one KV cache per branch.  Reading: node i of request r (T_r nodes, prefix P_r cached
slots) sees logical slots 0..P_r-1 and P_r + a for every a that is i or an ancestor of i; the
caller has written node a's K/V to logical slot P_r + a.  Logical slot s lives in physical block
block_table[r][s // bs] at offset s % bs.  Query head h reads KV head h // (H_q / H_kv).
Scale 1/sqrt(d); lse is the natural log of the sum of exp(scaled scores).
"""
import numpy as np

from .tree import ancestors_or_self

BAD_BLOCK = 32


def _gather(cache, table_row, slots, h, bs):
    blocks = table_row[np.asarray(slots) // bs]
    return cache[blocks, h, np.asarray(slots) % bs, :]


def visible_slots(par, i, P):
    """Logical KV slots node i attends to: the prefix, then its own path in the tree."""
    return list(range(P)) + sorted(P + a for a in ancestors_or_self(par, i))


def tree_attention(q, k_cache, v_cache, block_table, prefix_len, node_offset, parent, bs,
                   scale=None, rows=None):
    """q: [N, H_q, d]; k_cache / v_cache: [num_blocks, H_kv, bs, d] (one layer), any real dtype.

    Returns dict(o [N, H_q, d] fp64, lse [N, H_q] fp64, status [B]); entries that were not
    computed (rows not requested, bad requests) are NaN.  `rows`, if given, is an iterable of
    (global node, query head) pairs to compute; otherwise every pair is computed.
    """
    q = np.asarray(q, dtype=np.float64)
    kc = np.asarray(k_cache, dtype=np.float64)
    vc = np.asarray(v_cache, dtype=np.float64)
    table = np.asarray(block_table, dtype=np.int64)
    node_offset = np.asarray(node_offset, dtype=np.int64)
    parent = np.asarray(parent, dtype=np.int64)
    N, H_q, d = q.shape
    H_kv = kc.shape[1]
    G = H_q // H_kv
    num_blocks = kc.shape[0]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    B = len(node_offset) - 1
    o_out = np.full((N, H_q, d), np.nan)
    lse_out = np.full((N, H_q), np.nan)
    status = np.zeros(B, dtype=np.int64)
    owner = np.zeros(N, dtype=np.int64)
    for r in range(B):
        owner[node_offset[r]:node_offset[r + 1]] = r
    if rows is None:
        rows = [(n, h) for n in range(N) for h in range(H_q)]
    by_req = {}
    for n, h in rows:
        by_req.setdefault(int(owner[n]), []).append((int(n), int(h)))
    for r, items in sorted(by_req.items()):
        o, T, P = int(node_offset[r]), int(node_offset[r + 1] - node_offset[r]), int(prefix_len[r])
        nblk = -(-(P + T) // bs)
        if np.any(table[r, :nblk] < 0) or np.any(table[r, :nblk] >= num_blocks):
            status[r] |= BAD_BLOCK
            continue
        par = parent[o:o + T]
        for n, h in items:
            i = n - o
            slots = visible_slots(par, i, P)
            K = _gather(kc, table[r], slots, h // G, bs)
            Vv = _gather(vc, table[r], slots, h // G, bs)
            s = (K @ q[n, h]) * scale
            m = s.max()
            w = np.exp(s - m)
            z = w.sum()
            o_out[n, h] = (w @ Vv) / z
            lse_out[n, h] = m + np.log(z)
    return dict(o=o_out, lse=lse_out, status=status)
