"""Oracle: flattened draft tree -> ancestor mask, depth, position ids, internal-node flags.

Follows "投机推理算法的常见优化手段" (cnblogs zrq96), section 草稿树的验证——树形掩码: the tree is
flattened in BFS order ([root, A, B, C, D, E] in the page's figure) and each token may only see
its ancestors; the page's mask table has one row per query token and a 1 in column j exactly
when j is the row itself or one of its ancestors (root row: only root; C row: root, A, C).  The
same section says mask, KV cache and position ids must all adapt to the tree; position id =
prefix length + depth is the reading used here (depth(root) = 0).
"""
import numpy as np

BAD_PARENT = 1
BAD_SIZE = 2


def ancestors_or_self(par, i):
    """Walk the parent chain from local node i up to the root: [i, parent(i), ..., 0]."""
    out = []
    j = i
    while j != -1:
        out.append(j)
        j = int(par[j])
    return out


def tree_build(parent, node_offset, prefix_len, T_max):
    """Per request r (nodes node_offset[r] .. node_offset[r+1]-1, parent given as local index):

    returns dict(depth[N], pos_id[N], is_internal[N] (bool), mask[r] (bool [T_r, T_r] with
    mask[i, j] = j is i or an ancestor of i), status[B]).  A request whose tree is not a valid
    BFS/topological parent array (parent[0] = -1, 0 <= parent[i] < i) gets BAD_PARENT; one with
    T_r < 1 or T_r > T_max gets BAD_SIZE; its outputs are left at -1 / empty.
    """
    parent = np.asarray(parent, dtype=np.int64)
    node_offset = np.asarray(node_offset, dtype=np.int64)
    B = len(node_offset) - 1
    N = int(node_offset[-1])
    depth = np.full(N, -1, dtype=np.int64)
    pos_id = np.full(N, -1, dtype=np.int64)
    is_internal = np.zeros(N, dtype=bool)
    masks = [None] * B
    status = np.zeros(B, dtype=np.int64)
    for r in range(B):
        o, T = int(node_offset[r]), int(node_offset[r + 1] - node_offset[r])
        if T < 1 or T > T_max:
            status[r] |= BAD_SIZE
            continue
        par = parent[o:o + T]
        if par[0] != -1 or any(not (0 <= par[i] < i) for i in range(1, T)):
            status[r] |= BAD_PARENT
            continue
        M = np.zeros((T, T), dtype=bool)
        for i in range(T):
            chain = ancestors_or_self(par, i)
            for j in chain:
                M[i, j] = True
            depth[o + i] = len(chain) - 1
            pos_id[o + i] = int(prefix_len[r]) + depth[o + i]
        for i in range(1, T):
            is_internal[o + par[i]] = True
        masks[r] = M
    return dict(depth=depth, pos_id=pos_id, is_internal=is_internal, mask=masks, status=status)
