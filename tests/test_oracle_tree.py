"""Pins for oracle.tree: the page's worked mask table, the printed node counts, chains."""
import numpy as np
import pytest

from oracle import tree as OT
from speculative_decoding_draft_tree_gb300 import workloads as W
from conftest import golden_path


def _read_mask_fixture():
    parent, rows = None, []
    with open(golden_path("tree6_mask.txt"), encoding="utf-8") as f:
        lines = f.read().splitlines()
    for line in lines:
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split()
        if parts[0] == "parent":
            parent = [int(x) for x in parts[1:]]
        else:
            rows.append([int(x) for x in parts[1:]])
    return parent, np.array(rows, dtype=bool)


def test_page_mask_table_reproduced_exactly():
    parent, want = _read_mask_fixture()
    out = OT.tree_build(parent, [0, 6], [0], T_max=8)
    assert out["status"][0] == 0
    np.testing.assert_array_equal(out["mask"][0], want)
    # figure: root, A, B have children; C, D, E are leaves; depths 0, 1, 1, 2, 2, 2
    assert out["is_internal"].tolist() == [True, True, True, False, False, False]
    assert out["depth"].tolist() == [0, 1, 1, 2, 2, 2]


def test_position_ids_are_prefix_plus_depth():
    parent, _ = _read_mask_fixture()
    out = OT.tree_build(parent + parent, [0, 6, 12], [100, 7], T_max=8)
    assert out["pos_id"].tolist() == [100, 101, 101, 102, 102, 102, 7, 8, 8, 9, 9, 9]


def _read_counts():
    rows = {}
    with open(golden_path("node_counts.txt"), encoding="utf-8") as f:
        lines = f.read().splitlines()
    for line in lines:
        if line.startswith("#") or not line.strip():
            continue
        name, ks, per_depth, total, leaves = [x.strip() for x in line.split("|")]
        rows[name] = ([int(x) for x in ks.split()], [int(x) for x in per_depth.split()],
                      int(total), int(leaves))
    return rows


@pytest.mark.parametrize("name", ["medusa", "specinfer"])
def test_printed_node_counts(name):
    ks, per_depth, total, leaves = _read_counts()[name]
    parent = W.cartesian_parents(ks)
    T = len(parent)
    out = OT.tree_build(parent, [0, T], [0], T_max=256)
    depth = out["depth"]
    assert T - 1 == total
    assert [int((depth == l).sum()) for l in range(1, len(ks) + 1)] == per_depth
    assert int((~out["is_internal"]).sum()) == leaves


def test_chain_mask_is_lower_triangular():
    T = 7
    out = OT.tree_build(W.chain_parents(T), [0, T], [0], T_max=8)
    np.testing.assert_array_equal(out["mask"][0], np.tril(np.ones((T, T), dtype=bool)))
    assert out["depth"].tolist() == list(range(T))
    assert out["is_internal"].tolist() == [True] * (T - 1) + [False]   # all but the last


def test_invalid_trees_flagged():
    # parent[i] >= i, root with a parent, oversize tree
    out = OT.tree_build([-1, 0, 3, 1] + [0, 0] + [-1] * 3, [0, 4, 6, 9], [0, 0, 0], T_max=2)
    assert out["status"][0] & OT.BAD_SIZE  # T = 4 > T_max = 2
    out = OT.tree_build([-1, 0, 3, 1], [0, 4], [0], T_max=8)
    assert out["status"][0] == OT.BAD_PARENT
    out = OT.tree_build([0, 0], [0, 2], [0], T_max=8)
    assert out["status"][0] == OT.BAD_PARENT
    out = OT.tree_build([], [0, 0], [0], T_max=8)
    assert out["status"][0] == OT.BAD_SIZE
    # the size bound is inclusive: T = T_max is built, T = T_max + 1 is refused
    out = OT.tree_build([-1, 0, 1] + [-1, 0], [0, 3, 5], [0, 0], T_max=2)
    assert out["status"].tolist() == [OT.BAD_SIZE, 0]
