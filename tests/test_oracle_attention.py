"""Pins for oracle.attention against library scaled-dot-product attention (torch, fp64).

Special cases that reduce to a textbook routine: a single tree token (T = 1) is plain decode
attention over prefix + root; a chain tree is causal attention over prefix + chain; any tree node
equals causal attention over prefix + its own root-to-node path (tree-based and sequence-based
decoding agree, m.haoling.cc section 5.2); GQA maps query head h to KV head h // G.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as OA
from speculative_decoding_draft_tree_gb300 import workloads as W


def _dense(kc, vc, table, slots, h, bs):
    blocks = table[np.asarray(slots) // bs]
    return kc[blocks, h, np.asarray(slots) % bs], vc[blocks, h, np.asarray(slots) % bs]


def _case(parents_per_req, prefix, H_q=4, H_kv=2, d=16, bs=4, seed=0, permute=True):
    rng = np.random.default_rng(seed)
    B = len(parents_per_req)
    sizes = [len(p) for p in parents_per_req]
    no = np.concatenate([[0], np.cumsum(sizes)])
    N = int(no[-1])
    need = [-(-(prefix[r] + sizes[r]) // bs) for r in range(B)]
    nb = sum(need) + 3
    perm = rng.permutation(nb) if permute else np.arange(nb)
    table = np.full((B, max(need)), -1)
    pos = 0
    for r in range(B):
        table[r, :need[r]] = perm[pos:pos + need[r]]
        pos += need[r]
    q = rng.normal(size=(N, H_q, d))
    kc = rng.normal(size=(nb, H_kv, bs, d))
    vc = rng.normal(size=(nb, H_kv, bs, d))
    parent = np.concatenate([np.asarray(p) for p in parents_per_req])
    return q, kc, vc, table, np.asarray(prefix), no, parent


def _sdpa_last_row(qv, K, Vv, causal_len):
    """library attention of one query (the last of a causal sequence) over K, V (fp64)."""
    qt = torch.tensor(qv, dtype=torch.float64).view(1, 1, 1, -1)
    kt = torch.tensor(K, dtype=torch.float64).view(1, 1, causal_len, -1)
    vt = torch.tensor(Vv, dtype=torch.float64).view(1, 1, causal_len, -1)
    return F.scaled_dot_product_attention(qt, kt, vt).view(-1).numpy()


def test_single_token_is_decode_attention():
    q, kc, vc, table, P, no, parent = _case([[-1], [-1]], [13, 1])
    out = OA.tree_attention(q, kc, vc, table, P, no, parent, bs=4)
    for r in range(2):
        for h in range(4):
            K, Vv = _dense(kc, vc, table[r], list(range(P[r] + 1)), h // 2, 4)
            ref = _sdpa_last_row(q[no[r], h], K, Vv, P[r] + 1)
            np.testing.assert_allclose(out["o"][no[r], h], ref, rtol=1e-12, atol=1e-12)
            # lse: the natural log of the sum of exp(scaled scores), by the library's logsumexp
            s = torch.tensor(K @ q[no[r], h] / np.sqrt(q.shape[2]))
            assert abs(out["lse"][no[r], h] - float(torch.logsumexp(s, 0))) < 1e-12


def test_explicit_scale():
    # a caller's own softmax scale replaces 1/sqrt(d): library attention with the same scale
    q, kc, vc, table, P, no, parent = _case([[-1]], [9])
    out = OA.tree_attention(q, kc, vc, table, P, no, parent, bs=4, scale=0.3)
    for h in range(4):
        K, Vv = _dense(kc, vc, table[0], list(range(P[0] + 1)), h // 2, 4)
        ref = F.scaled_dot_product_attention(
            torch.tensor(q[0, h]).view(1, 1, 1, -1), torch.tensor(K).view(1, 1, P[0] + 1, -1),
            torch.tensor(Vv).view(1, 1, P[0] + 1, -1), scale=0.3).view(-1).numpy()
        np.testing.assert_allclose(out["o"][0, h], ref, rtol=1e-12, atol=1e-12)


def test_kv_length_one():
    q, kc, vc, table, P, no, parent = _case([[-1]], [0])
    out = OA.tree_attention(q, kc, vc, table, P, no, parent, bs=4)
    K, Vv = _dense(kc, vc, table[0], [0], 0, 4)
    np.testing.assert_allclose(out["o"][0, 0], Vv[0], rtol=1e-13)
    np.testing.assert_allclose(out["lse"][0, 0], K[0] @ q[0, 0] / 4.0, rtol=1e-13)


def test_chain_is_causal_attention():
    T, P = 6, 9
    q, kc, vc, table, Pv, no, parent = _case([W.chain_parents(T)], [P], H_q=2, H_kv=2)
    out = OA.tree_attention(q, kc, vc, table, Pv, no, parent, bs=4)
    for h in range(2):
        K, Vv = _dense(kc, vc, table[0], list(range(P + T)), h, 4)
        qt = torch.zeros(1, 1, P + T, q.shape[2], dtype=torch.float64)
        qt[0, 0, P:] = torch.tensor(q[:, h])
        ref = F.scaled_dot_product_attention(
            qt, torch.tensor(K).view(1, 1, P + T, -1), torch.tensor(Vv).view(1, 1, P + T, -1),
            is_causal=True)[0, 0, P:].numpy()
        np.testing.assert_allclose(out["o"][:, h], ref, rtol=1e-12, atol=1e-12)


def test_tree_node_equals_sequence_over_its_path():
    parents = [W.cartesian_parents((2, 3)), W.cartesian_parents((3, 1, 2))]
    q, kc, vc, table, P, no, parent = _case(parents, [5, 16], H_q=6, H_kv=3, d=8)
    out = OA.tree_attention(q, kc, vc, table, P, no, parent, bs=4)
    for r, par in enumerate(parents):
        for i in range(len(par)):
            path = []
            j = i
            while j != -1:
                path.append(j)
                j = par[j]
            seq = list(range(P[r])) + [P[r] + a for a in reversed(path)]
            for h in range(6):
                K, Vv = _dense(kc, vc, table[r], seq, h // 2, 4)
                ref = _sdpa_last_row(q[no[r] + i, h], K, Vv, len(seq))
                np.testing.assert_allclose(out["o"][no[r] + i, h], ref, rtol=1e-12, atol=1e-12)


def test_paging_is_invisible():
    parents = [W.cartesian_parents((2, 2)), W.chain_parents(3)]
    a = _case(parents, [7, 31], seed=3, permute=True)
    q, kc, vc, table, P, no, parent = a
    out_paged = OA.tree_attention(q, kc, vc, table, P, no, parent, bs=4)
    # rebuild the same logical cache contiguously
    B = 2
    need = table.shape[1]
    kc2 = np.zeros((B * need, kc.shape[1], 4, kc.shape[3]))
    vc2 = np.zeros_like(kc2)
    t2 = np.full_like(table, -1)
    for r in range(B):
        for j in range(need):
            if table[r, j] >= 0:
                kc2[r * need + j] = kc[table[r, j]]
                vc2[r * need + j] = vc[table[r, j]]
                t2[r, j] = r * need + j
    out_flat = OA.tree_attention(q, kc2, vc2, t2, P, no, parent, bs=4)
    np.testing.assert_array_equal(out_paged["o"], out_flat["o"])


def test_bad_block_flagged():
    q, kc, vc, table, P, no, parent = _case([[-1, 0]], [6])
    table[0, 1] = kc.shape[0]
    out = OA.tree_attention(q, kc, vc, table, P, no, parent, bs=4)
    assert out["status"][0] == OA.BAD_BLOCK
    assert np.isnan(out["o"]).all()
    # a partly filled last block (blocks of 4; prefix 4 puts the two nodes in slots 4, 5 of
    # block 1, prefix 3 puts slot 4 alone there): a bad id there is still found
    for P in (4, 3):
        q, kc, vc, table, Pv, no, parent = _case([[-1, 0]], [P])
        table[0, 1] = -1
        out = OA.tree_attention(q, kc, vc, table, Pv, no, parent, bs=4)
        assert out["status"][0] == OA.BAD_BLOCK, P
