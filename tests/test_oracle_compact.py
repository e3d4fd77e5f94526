"""Pins for oracle.compact: after compaction the cache equals the cache that sequential decoding
of the accepted path would have written (root, then each accepted draft, one slot after another),
the prefix is untouched and the committed length is P + n_acc + 1."""
import numpy as np
import pytest

from oracle import compact as OC
from speculative_decoding_draft_tree_gb300 import workloads as W


def _random_case(rng, B=4, L=2, H=3, d=4, bs=4):
    parents, paths, P = [], [], []
    for r in range(B):
        ks = [int(x) for x in rng.integers(1, 4, size=rng.integers(1, 4))]
        par = W.cartesian_parents(ks)
        parents.append(par)
        node = int(rng.integers(0, len(par)))      # accept the root-to-node path
        path = []
        while node != -1:
            path.append(node)
            node = par[node]
        paths.append(path[::-1])
        P.append(int(rng.integers(0, 20)))
    need = [-(-(P[r] + len(parents[r])) // bs) for r in range(B)]
    nb = sum(need) + 2
    perm = rng.permutation(nb)
    table = np.full((B, max(need)), -1)
    pos = 0
    for r in range(B):
        table[r, :need[r]] = perm[pos:pos + need[r]]
        pos += need[r]
    # every (layer, block, head, offset) holds a distinct code so moves are traceable
    k = rng.normal(size=(L, nb, H, bs, d))
    v = rng.normal(size=(L, nb, H, bs, d))
    return parents, paths, P, table, k, v, bs


def _slot(cache, table_row, s, bs):
    return cache[:, table_row[s // bs], :, s % bs, :]


def test_compaction_equals_sequential_decoding():
    rng = np.random.default_rng(0)
    for trial in range(20):
        parents, paths, P, table, k, v, bs = _random_case(rng)
        B = len(parents)
        max_path = 8
        n_acc = [len(p) - 1 for p in paths]
        out = OC.kv_compact(k, v, table, P, paths, n_acc, bs, max_path)
        for r in range(B):
            # sequential decoding writes node path[d]'s K/V into slot P + d
            for dd, node in enumerate(paths[r]):
                np.testing.assert_array_equal(_slot(out["k"], table[r], P[r] + dd, bs),
                                              _slot(k, table[r], P[r] + node, bs))
                np.testing.assert_array_equal(_slot(out["v"], table[r], P[r] + dd, bs),
                                              _slot(v, table[r], P[r] + node, bs))
                assert tuple(out["slot_map"][r, dd]) == (P[r] + node, P[r] + dd)
            for s in range(P[r]):   # the prefix is never touched
                np.testing.assert_array_equal(_slot(out["k"], table[r], s, bs),
                                              _slot(k, table[r], s, bs))
            assert out["new_kv_len"][r] == P[r] + n_acc[r] + 1
            assert out["blocks_in_use"][r] == -(-(P[r] + n_acc[r] + 1) // bs)
            assert (out["slot_map"][r, n_acc[r] + 1:] == -1).all()


def test_rejected_request_rolls_back_everything():
    rng = np.random.default_rng(1)
    parents, paths, P, table, k, v, bs = _random_case(rng, B=2)
    out = OC.kv_compact(k, v, table, P, paths, [-1, len(paths[1]) - 1], bs, 8)
    assert out["new_kv_len"][0] == P[0]
    assert (out["slot_map"][0] == -1).all()
    out2 = OC.kv_compact(k, v, table, P, paths, [len(p) - 1 for p in paths], bs, 8, status=[4, 0])
    assert out2["new_kv_len"][0] == P[0]


def test_bad_block_flagged():
    rng = np.random.default_rng(2)
    parents, paths, P, table, k, v, bs = _random_case(rng, B=1)
    table[0, :] = k.shape[1] + 5
    out = OC.kv_compact(k, v, table, P, paths, [len(paths[0]) - 1], bs, 8)
    assert out["status"][0] == OC.BAD_BLOCK
    np.testing.assert_array_equal(out["k"], k)
    # rolled back: the committed length and the blocks in use are the prefix's
    assert out["new_kv_len"][0] == P[0] and out["blocks_in_use"][0] == -(-P[0] // bs)
