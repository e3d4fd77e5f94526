"""Helpers comparing the CUDA path (through the C-ABI) with the CPU oracle.

Bars (from the verification step's contract):
  * bit-exact: tree outputs, accepted lengths, accepted token ids, paths, rejection counts,
    compaction slot maps / lengths / moved cache rows, request status bits;
  * the only exception: a ratio test with |u - a| < 1e-6 or a resampled token whose uniform lies
    within 1e-6 of a CDF boundary (fp32 on the GPU cannot resolve fp64 closer than that); such
    a divergence exempts the rest of that request and is counted in TALLY; the whole suite's
    count must stay below 1e-5 of its draws (tests/test_zy_exemption_tally.py checks it after
    the parity tests);
  * attention: 1e-5 relative for fp32, 2e-2 absolute for bf16.
"""
import numpy as np
import torch

from oracle import attention as OA
from oracle import compact as OC
from oracle import tree as OT
from oracle import verify as OV

BAND = 1e-6
# draws checked and near-boundary exemptions over every check_verify call of the session
TALLY = {"draws": 0, "exempt": 0, "calls": 0}


def np_(t):
    return t.detach().cpu().numpy()


def f32(t):
    """Logit / probability rows as float32 numpy (bf16 values are exact in fp32)."""
    return t.detach().float().cpu().numpy()


def snapshot(w):
    return dict(parent=np_(w.parent), node_offset=np_(w.node_offset), prefix_len=np_(w.prefix_len),
                tokens=np_(w.tokens), draft_row=np_(w.draft_row), uniforms=np_(w.uniforms),
                block_table=np_(w.block_table))


# ---------------------------------------------------------------------------------- tree
def check_tree(w, step, snap):
    orc = OT.tree_build(snap["parent"], snap["node_offset"], snap["prefix_len"], w.T_max)
    st = np_(step.req_status)
    assert (st & 3).tolist() == orc["status"].tolist()
    depth, pos, internal = np_(step.depth), np_(step.pos_id), np_(step.is_internal)
    anc = np_(step.anc_mask).view(np.uint32)
    no = snap["node_offset"]
    for r in range(w.B):
        if orc["status"][r]:
            continue
        o, T = no[r], no[r + 1] - no[r]
        assert depth[o:o + T].tolist() == orc["depth"][o:o + T].tolist()
        assert pos[o:o + T].tolist() == orc["pos_id"][o:o + T].tolist()
        assert internal[o:o + T].astype(bool).tolist() == orc["is_internal"][o:o + T].tolist()
        bits = np.zeros((T, T), dtype=bool)
        for i in range(T):
            for j in range(T):
                bits[i, j] = (anc[o + i, j >> 5] >> np.uint32(j & 31)) & 1
        np.testing.assert_array_equal(bits, orc["mask"][r])
    return orc


# ---------------------------------------------------------------------------------- verify
def oracle_verify(w, snap, sibling_rule=OV.SIBLING_RESIDUAL, target=None, draft=None):
    target = f32(w.target) if target is None else target
    draft = f32(w.draft) if draft is None else draft
    return OV.verify(target, draft, w.draft_kind, snap["draft_row"], snap["tokens"],
                     snap["parent"], snap["node_offset"], snap["uniforms"], w.tau, w.V,
                     w.max_path, sibling_rule=sibling_rule, T_max=w.T_max)


def _near(events, node):
    for e in events:
        if e[1] != node:
            continue
        if e[0] == "test" and abs(e[4] - e[3]) < BAND:
            return True
        if e[0] == "sample" and e[3] < BAND:
            return True
    return False


def check_verify(w, step, orc, status_mask=~0):
    """Returns (draws, exempt)."""
    st = np_(step.req_status)
    out_len, n_acc = np_(step.out_len), np_(step.n_acc)
    path, toks, rej = np_(step.path), np_(step.out_tokens), np_(step.rejections)
    draws = exempt = 0
    for r in range(w.B):
        assert int(st[r]) & status_mask == int(orc["status"][r]) & status_mask, (r, st[r], orc["status"][r])
        if orc["status"][r]:
            assert out_len[r] == 0 and n_acc[r] == -1
            assert (path[r] == -1).all() and (toks[r] == -1).all()
            continue
        draws += max(1, len(orc["events"][r]))
        g_path = path[r, :n_acc[r] + 1].tolist() if n_acc[r] >= 0 else []
        g_tok = toks[r, :out_len[r]].tolist()
        if g_path == orc["path"][r] and g_tok == orc["out_tokens"][r]:
            assert rej[r] == orc["rejections"][r], (r, rej[r], orc["rejections"][r])
            assert (path[r, n_acc[r] + 1:] == -1).all() and (toks[r, out_len[r]:] == -1).all()
            continue
        # first divergence: the last common node of the two paths
        k = 0
        while k < min(len(g_path), len(orc["path"][r])) and g_path[k] == orc["path"][r][k]:
            k += 1
        node = orc["path"][r][k - 1]
        assert _near(orc["events"][r], node), (
            f"request {r}: GPU path {g_path} tokens {g_tok} vs oracle {orc['path'][r]} "
            f"{orc['out_tokens'][r]} (events {orc['events'][r]})")
        exempt += 1
    TALLY["draws"] += draws
    TALLY["exempt"] += exempt
    TALLY["calls"] += 1
    return draws, exempt


# ---------------------------------------------------------------------------------- compact
def tree_region_blocks(w, snap, r, n_slots=None):
    P = int(snap["prefix_len"][r])
    T = int(snap["node_offset"][r + 1] - snap["node_offset"][r])
    lo, hi = P // w.bs, (P + T - 1) // w.bs
    return [int(b) for b in snap["block_table"][r, lo:hi + 1]], lo


def cache_region(cache, w, snap, requests):
    """Copy of the cache blocks that hold the tree slots of `requests`: {r: [L, nb, H, bs, d]}."""
    out = {}
    for r in requests:
        blocks, _ = tree_region_blocks(w, snap, r)
        out[r] = cache[:, blocks].float().cpu().numpy()
    return out


def check_compact(w, step, snap, k_before, v_before):
    """k_before / v_before: cache_region() snapshots taken before spec_kv_compact ran."""
    st = np_(step.req_status)
    n_acc, path = np_(step.n_acc), np_(step.path)
    new_len, smap, biu = np_(step.new_kv_len), np_(step.slot_map), np_(step.blocks_in_use)
    k_after = cache_region(w.k_cache, w, snap, list(k_before.keys()))
    v_after = cache_region(w.v_cache, w, snap, list(v_before.keys()))
    for r in range(w.B):
        P = int(snap["prefix_len"][r])
        if r not in k_before:
            continue
        blocks, lo = tree_region_blocks(w, snap, r)
        nb = len(blocks)
        table = np.full((1, lo + nb), -1)
        table[0, lo:] = np.arange(nb)
        orc = OC.kv_compact(k_before[r], v_before[r], table, [P], [path[r].tolist()],
                            [int(n_acc[r])], w.bs, w.max_path, status=[int(st[r])])
        assert new_len[r] == orc["new_kv_len"][0]
        assert biu[r] == orc["blocks_in_use"][0]
        np.testing.assert_array_equal(smap[r], orc["slot_map"][0])
        np.testing.assert_array_equal(k_after[r], orc["k"])
        np.testing.assert_array_equal(v_after[r], orc["v"])


# ---------------------------------------------------------------------------------- attention
def check_attention(w, step, snap, rows=None, k_cache_layer0=None, v_cache_layer0=None):
    """Compare O (and LSE) with the oracle on `rows` ((node, head) pairs; all when None)."""
    st = np_(step.req_status)
    kc = (w.k_cache[0] if k_cache_layer0 is None else k_cache_layer0)
    vc = (w.v_cache[0] if v_cache_layer0 is None else v_cache_layer0)
    if rows is None:
        rows = [(n, h) for n in range(w.N) for h in range(w.H_q)]
    owner = np.searchsorted(snap["node_offset"], np.arange(w.N), side="right") - 1
    rows = [(n, h) for (n, h) in rows if st[owner[n]] == 0]
    # gather only the blocks the sampled requests use
    reqs = sorted(set(int(owner[n]) for n, _ in rows))
    q = f32(w.q).astype(np.float64)
    o_gpu = f32(step.o)
    lse_gpu = None if step.lse is None else np_(step.lse)
    tol_abs, tol_rel = (2e-2, 0.0) if w.dtype == "bf16" else (0.0, 1e-5)
    worst = 0.0
    for r in reqs:
        P = int(snap["prefix_len"][r])
        o0, o1 = int(snap["node_offset"][r]), int(snap["node_offset"][r + 1])
        nblk = -(-(P + o1 - o0) // w.bs)
        blocks = snap["block_table"][r, :nblk].astype(np.int64)
        kr = kc[torch.as_tensor(blocks, device=kc.device)].float().cpu().numpy()
        vr = vc[torch.as_tensor(blocks, device=vc.device)].float().cpu().numpy()
        table = np.arange(nblk)[None, :]
        sub_rows = [(n - o0, h) for (n, h) in rows if o0 <= n < o1]
        orc = OA.tree_attention(q[o0:o1], kr, vr, table, [P], [0, o1 - o0],
                                snap["parent"][o0:o1], w.bs, rows=sub_rows)
        for (i, h) in sub_rows:
            ref = orc["o"][i, h]
            got = o_gpu[o0 + i, h].astype(np.float64)
            if tol_rel:
                np.testing.assert_allclose(got, ref, rtol=tol_rel, atol=1e-6)
            else:
                np.testing.assert_allclose(got, ref, atol=tol_abs, rtol=0)
            worst = max(worst, float(np.abs(got - ref).max()))
            if lse_gpu is not None:
                np.testing.assert_allclose(lse_gpu[o0 + i, h], orc["lse"][i, h], rtol=1e-5,
                                           atol=1e-4)
    return worst
