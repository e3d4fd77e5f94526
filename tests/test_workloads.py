"""The seeded input generators: Philox known answers, shapes of the five workloads."""
import numpy as np
import pytest

from speculative_decoding_draft_tree_gb300 import workloads as W


def test_philox_known_answers():
    # Random123 known-answer vectors for philox4x32_10
    cases = [
        ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
        ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
        ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
         (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
    ]
    for ctr, key, want in cases:
        got = W.philox4x32_10(np.array([ctr], dtype=np.uint32), key)[0]
        assert tuple(int(x) for x in got) == want


def test_uniforms_in_unit_interval_and_exact():
    u = W.node_uniforms(10000, seed=0)
    assert u.dtype == np.float32 and (u >= 0).all() and (u < 1).all()
    assert np.all(u.astype(np.float64) * 2 ** 24 == np.round(u.astype(np.float64) * 2 ** 24))
    assert abs(u.mean() - 0.5) < 0.01


@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5])
def test_small_configs_are_consistent(cid):
    w = W.make_config(cid, scale="small")
    no = w.node_offset.numpy()
    par = w.parent.numpy()
    assert no[0] == 0 and no[-1] == w.N
    assert w.target.shape[0] == w.N and w.target.shape[1] >= w.V
    assert (w.target.shape[1] * w.target.element_size()) % 16 == 0
    assert w.q.shape == (w.N, w.H_q, w.d)
    for r in range(w.B):
        T = no[r + 1] - no[r]
        assert 1 <= T <= w.T_max
        loc = par[no[r]:no[r + 1]]
        assert loc[0] == -1 and all(0 <= loc[i] < i for i in range(1, T))
        need = -(-(int(w.prefix_len[r]) + T) // w.bs)
        assert (w.block_table[r, :need] >= 0).all()
    # every node with children has a draft row
    has_child = np.zeros(w.N, dtype=bool)
    for r in range(w.B):
        for i in range(1, no[r + 1] - no[r]):
            has_child[no[r] + par[no[r] + i]] = True
    assert (w.draft_row.numpy()[has_child] >= 0).all()


def test_eagle2_echo_budget_and_closure():
    w = W.make_config(5, scale="small")
    assert w.N == 150 and len(w.tree_sizes()) == 4
    assert max(w.tree_sizes()) <= 1 + 5 + 25 * 7


def test_generation_is_deterministic():
    a = W.make_config(4, scale="small")
    b = W.make_config(4, scale="small")
    assert (a.tokens == b.tokens).all() and (a.target == b.target).all()
    assert (a.k_cache == b.k_cache).all() and (a.uniforms == b.uniforms).all()


def test_lookahead_shape_matches_the_oracles_mask():
    """The generator's lookahead trees are the oracle's (built from the page's mask rules)."""
    from oracle import lookahead as OL
    for W_, N_, G_ in [(5, 4, 5), (15, 5, 15), (10, 5, 10), (7, 5, 7), (3, 3, 2), (6, 2, 0)]:
        assert W.lookahead_parents(W_, N_, G_) == OL.lookahead_parents(W_, N_, G_).tolist()
