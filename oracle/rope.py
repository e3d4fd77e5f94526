"""Oracle: rotary position embedding at the tree's position ids, and the tree K/V written into
its paged cache slots -- the step just before tree attention.

Follows "投机推理算法的常见优化手段" (cnblogs zrq96), section 草稿树的验证——树形掩码: the forward
call over the draft tree takes the tree, its mask, its position ids and the KV cache, and mask,
KV cache and position ids must all follow the tree.  The pages do not say how a position id
enters the model.  Reading: rotary position embedding (Su et al., "RoFormer: Enhanced
Transformer with Rotary Position Embedding", 2021, section 3.2), the position scheme of the
model families these workloads are shaped after, applied to q and k at position id
pos = prefix length + depth, with the node's K/V then stored at logical slot prefix + (local
node index), where the attention step reads it.

RoPE at position m rotates pair j of a vector (j = 0 .. rotary_dim/2 - 1) by the angle
m * theta_j, theta_j = base ** (-2 j / rotary_dim):
    (a, b) -> (a cos(m theta_j) - b sin(m theta_j), a sin(m theta_j) + b cos(m theta_j)).
Pair j is (x[2j], x[2j+1]) in the interleaved layout (the paper's) and (x[j], x[j + rotary_dim/2])
in the half-split layout used by LLaMA-family checkpoints.  Components past rotary_dim are not
rotated.  Everything here is fp64.
"""
import numpy as np

BAD_BLOCK = 32


def pair_indices(rotary_dim, interleaved):
    """The (a, b) component indices of every rotated pair, in pair order j."""
    half = rotary_dim // 2
    if interleaved:
        return [(2 * j, 2 * j + 1) for j in range(half)]
    return [(j, j + half) for j in range(half)]


def rope(x, pos, base=10000.0, rotary_dim=None, interleaved=False):
    """x: [..., d] (any real dtype); pos: integer array broadcastable to x.shape[:-1].
    Returns fp64 [..., d]: x with pair j of its first rotary_dim components rotated by
    pos * base ** (-2 j / rotary_dim)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    rotary_dim = d if rotary_dim is None else int(rotary_dim)
    if rotary_dim % 2 or not 0 < rotary_dim <= d:
        raise ValueError("rotary_dim must be even and in (0, d]")
    pos = np.broadcast_to(np.asarray(pos, dtype=np.float64), x.shape[:-1])
    out = x.copy()
    for j, (ia, ib) in enumerate(pair_indices(rotary_dim, interleaved)):
        theta = base ** (-2.0 * j / rotary_dim)
        ang = pos * theta
        c, s = np.cos(ang), np.sin(ang)
        a, b = x[..., ia], x[..., ib]
        out[..., ia] = a * c - b * s
        out[..., ib] = a * s + b * c
    return out


def tree_rope_kv_write(q, k_new, v_new, pos_id, node_offset, prefix_len, block_table, k_cache,
                       v_cache, base=10000.0, rotary_dim=None, interleaved=False,
                       req_status=None):
    """q [N, H_q, d], k_new / v_new [N, H_kv, d]; pos_id [N] (prefix + depth); caches
    [num_blocks, H_kv, bs, d] (one layer).  Node n = node_offset[r] + i of request r is rotated
    at pos_id[n]; its rotated k and its v go to logical slot prefix_len[r] + i, i.e. row
    (slot % bs) of physical block block_table[r][slot // bs].

    Requests with a nonzero req_status (from the tree build), a negative prefix length (no
    cache slots) or a negative pos_id are skipped.
    A request whose slot maps outside [0, num_blocks) gets BAD_BLOCK and none of its nodes are
    written.  Returns dict(q fp64 [N, H_q, d] (NaN where skipped), k_cache, v_cache (fp64
    copies with the slots written), status [B])."""
    q = np.asarray(q, dtype=np.float64)
    k_new = np.asarray(k_new, dtype=np.float64)
    v_new = np.asarray(v_new, dtype=np.float64)
    kc = np.array(k_cache, dtype=np.float64)
    vc = np.array(v_cache, dtype=np.float64)
    table = np.asarray(block_table, dtype=np.int64)
    node_offset = np.asarray(node_offset, dtype=np.int64)
    B = len(node_offset) - 1
    num_blocks, _, bs, _ = kc.shape
    status = np.zeros(B, dtype=np.int64) if req_status is None else np.array(req_status, np.int64)
    q_out = np.full(q.shape, np.nan)
    for r in range(B):
        if status[r]:
            continue
        o, T, P = int(node_offset[r]), int(node_offset[r + 1] - node_offset[r]), int(prefix_len[r])
        if P < 0:
            continue
        dest = []
        for i in range(T):
            slot = P + i
            lb = slot // bs
            blk = int(table[r, lb]) if lb < table.shape[1] else -1
            dest.append((blk, slot % bs))
        if any(not 0 <= b < num_blocks for b, _ in dest):
            status[r] |= BAD_BLOCK
            continue
        for i in range(T):
            n = o + i
            m = int(pos_id[n])
            if m < 0:
                continue
            q_out[n] = rope(q[n], m, base, rotary_dim, interleaved)
            blk, row = dest[i]
            kc[blk, :, row, :] = rope(k_new[n], m, base, rotary_dim, interleaved)
            vc[blk, :, row, :] = v_new[n]
    return dict(q=q_out, k_cache=kc, v_cache=vc, status=status)

