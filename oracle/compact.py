"""Oracle: KV commit / rollback of the accepted path.

Follows "推测解码 2026" (guijiagi.com), 工程实践中的考量 / KV Cache管理: the K/V of rejected
candidates must be rolled back, which paged (block) caches make cheap; and "【模型后训练与深度推理】9
推理加速：推测解码与级联推理" section 4: accepted tokens extend the prefix and the corrected token
seeds the next round while the cache is reused.  Reading: with the accepted path
path[0] = 0 (root), path[1..n_acc] (node indices), the committed cache after the round holds, in
logical slots P, P+1, ..., P+n_acc, the K/V that sequential decoding of root, then the accepted
drafts in order, would have written: new[P + d] = old[P + path[d]] (gather from the cache as it
was before compaction), for every layer, KV head, K and V.  new_kv_len = P + n_acc + 1; the
final (bonus / corrected) token has no K/V yet.  Slots past new_kv_len are released (not
cleared).  A request with a data error (or n_acc < 0) rolls the whole tree back:
new_kv_len = P and nothing is copied.
"""
import numpy as np

BAD_BLOCK = 32


def kv_compact(k_cache, v_cache, block_table, prefix_len, path, n_acc, bs, max_path,
               status=None):
    """k_cache / v_cache: [L, num_blocks, H_kv, bs, d].  path: list of lists (or [B, max_path]
    with -1 padding).  Returns dict(k, v (compacted copies), new_kv_len[B], slot_map[B, max_path,
    2] (src, dst logical slots, -1 padded), blocks_in_use[B], status[B])."""
    old_k = np.array(k_cache, copy=True)
    old_v = np.array(v_cache, copy=True)
    new_k = old_k.copy()
    new_v = old_v.copy()
    table = np.asarray(block_table, dtype=np.int64)
    B = table.shape[0]
    num_blocks = old_k.shape[1]
    status = np.zeros(B, dtype=np.int64) if status is None else np.array(status, dtype=np.int64)
    new_len = np.zeros(B, dtype=np.int64)
    slot_map = np.full((B, max_path, 2), -1, dtype=np.int64)
    blocks_in_use = np.zeros(B, dtype=np.int64)
    for r in range(B):
        P = int(prefix_len[r])
        na = int(n_acc[r])
        new_len[r] = P
        if status[r] or na < 0:
            blocks_in_use[r] = -(-P // bs)
            continue
        pr = [int(x) for x in path[r][: na + 1]]
        slots = [P + x for x in pr] + [P + dd for dd in range(na + 1)]
        blk = [table[r, s // bs] for s in slots]
        if any(b < 0 or b >= num_blocks for b in blk):
            status[r] |= BAD_BLOCK
            blocks_in_use[r] = -(-P // bs)
            continue
        for dd in range(na + 1):
            src, dst = P + pr[dd], P + dd
            slot_map[r, dd] = (src, dst)
            sb, so = table[r, src // bs], src % bs
            db, do = table[r, dst // bs], dst % bs
            new_k[:, db, :, do, :] = old_k[:, sb, :, so, :]
            new_v[:, db, :, do, :] = old_v[:, sb, :, so, :]
        new_len[r] = P + na + 1
        blocks_in_use[r] = -(-new_len[r] // bs)
    return dict(k=new_k, v=new_v, new_kv_len=new_len, slot_map=slot_map,
                blocks_in_use=blocks_in_use, status=status)
