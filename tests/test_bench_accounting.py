"""bench.py's algorithmic byte and flop counts, the numerators of its roofline fractions, against
brute force on the small workloads.

  * tree attention: the distinct key / value rows its requests must read (the union of every
    node's visible slots, from the oracle's visibility rule), Q read and O / LSE written once;
    its flops from every node's own visible keys;
  * RoPE + K/V write: the q, k and v rows the oracle's write reads and writes, counted from its
    outputs;
  * the compaction's share of a step: the cache slots the oracle's compaction changes, K and V
    read and written, every layer.
"""
import types

import numpy as np
import pytest
import torch

import bench
from oracle import attention as OA
from oracle import compact as OC
from oracle import rope as OR
from oracle import tree as OT
from oracle import verify as OV
from speculative_decoding_draft_tree_gb300 import workloads as W

CIDS = [1, 2, 3, 4, 5]


def _small(cid, **kw):
    return W.make_config(cid, scale="small", device="cpu", **kw)


def _es(w):
    return 2 if w.dtype == "bf16" else 4


def _trees(w):
    no, par, P = w.node_offset.numpy(), w.parent.numpy(), w.prefix_len.numpy()
    for r in range(w.B):
        o, T = int(no[r]), int(no[r + 1] - no[r])
        yield r, o, T, par[o:o + T], int(P[r])


@pytest.mark.parametrize("cid", CIDS)
def test_attention_bytes_are_the_distinct_rows_read(cid):
    w = _small(cid)
    kv_rows = 0
    for r, o, T, par, P in _trees(w):
        seen = set()
        for i in range(T):
            seen.update(OA.visible_slots(par, i, P))
        kv_rows += len(seen)
    es = _es(w)
    want = (kv_rows * w.H_kv * w.d * es * 2           # K and V, each row once per KV head
            + 2 * w.N * w.H_q * w.d * es              # Q read, O written
            + w.N * w.H_q * 4)                        # LSE (fp32) written
    assert bench.attention_bytes(w) == want


@pytest.mark.parametrize("cid", CIDS)
def test_attention_flops_count_each_nodes_visible_keys(cid):
    w = _small(cid)
    keys = sum(len(OA.visible_slots(par, i, P)) for r, o, T, par, P in _trees(w)
               for i in range(T))
    # q.k and p.v: 2 flops per multiply-add, head_dim of each per visible key and query head
    assert bench.attention_flops(w) == 2 * 2 * keys * w.H_q * w.d


@pytest.mark.parametrize("cid", [2, 3, 4])
def test_rope_bytes_are_the_rows_read_and_written(cid):
    w = _small(cid)
    tb = OT.tree_build(w.parent.numpy(), w.node_offset.numpy(), w.prefix_len.numpy(), w.T_max)
    k_new = torch.randn((w.N, w.H_kv, w.d), generator=torch.Generator().manual_seed(1)).numpy()
    v_new = torch.randn((w.N, w.H_kv, w.d), generator=torch.Generator().manual_seed(2)).numpy()
    kc = w.k_cache[0].float().numpy()
    vc = w.v_cache[0].float().numpy()
    out = OR.tree_rope_kv_write(w.q.float().numpy(), k_new, v_new, tb["pos_id"],
                                w.node_offset.numpy(), w.prefix_len.numpy(), w.block_table.numpy(),
                                kc, vc)
    assert not out["status"].any()
    q_rows = int((~np.isnan(out["q"]).any(axis=-1)).sum())          # (node, head) rows written
    k_rows = int((out["k_cache"] != kc).any(axis=-1).sum())         # cache rows written
    v_rows = int((out["v_cache"] != vc).any(axis=-1).sum())
    assert q_rows == w.N * w.H_q and k_rows == v_rows == w.N * w.H_kv
    # every row written was read once from its input
    assert bench.rope_bytes(w) == 2 * (q_rows + k_rows + v_rows) * w.d * _es(w)


@pytest.mark.parametrize("cid", [2, 3, 4, 5])
def test_step_bytes_compaction_share_is_the_slots_it_changes(cid):
    w = _small(cid, num_layers=2)
    no, V = w.node_offset.numpy(), w.V
    tb = OT.tree_build(w.parent.numpy(), no, w.prefix_len.numpy(), w.T_max)
    orc = OV.verify(w.target[:, :V].float().numpy(), w.draft[:, :V].float().numpy(), w.draft_kind,
                    w.draft_row.numpy(), w.tokens.numpy(), w.parent.numpy(), no,
                    w.uniforms.numpy(), w.tau, V, w.max_path, T_max=w.T_max)
    kc, vc = w.k_cache.float().numpy(), w.v_cache.float().numpy()
    comp = OC.kv_compact(kc, vc, w.block_table.numpy(), w.prefix_len.numpy(), orc["path"],
                         orc["n_acc"], w.bs, w.max_path, status=orc["status"])
    # cache slots (request, layer, KV head, logical slot) whose content the compaction changed
    changed = int((comp["k"] != kc).any(axis=-1).sum() + (comp["v"] != vc).any(axis=-1).sum())
    assert changed > 0 or cid == 2   # a chain's accepted path is already in place
    step = types.SimpleNamespace(is_internal=torch.from_numpy(tb["is_internal"].astype(np.uint8)),
                                 slot_map=torch.from_numpy(comp["slot_map"]))
    internal = tb["is_internal"]
    drows = len(set(w.draft_row.numpy()[internal].tolist())) if w.tau > 0 else 0
    ver = (int(internal.sum()) + drows + w.B * (2 if w.tau > 0 else 1)) * V * _es(w)
    comp_bytes = bench.step_bytes(w, step) - bench.attention_bytes(w) - ver
    # each changed K or V row was read from its source slot and written once
    assert comp_bytes == 2 * changed * w.d * _es(w)
