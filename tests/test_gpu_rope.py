"""GPU <-> oracle parity of spec_tree_rope_kv_write (rotary embedding at the tree's position ids
and the tree K/V written into its paged slots) through the C-ABI.

Bars, from the arithmetic: the GPU forms and reduces each angle in fp64 and rotates in fp32, so
before the final rounding its value differs from the fp64 oracle by at most
eps = 1e-6 * (|a| + |b|) for a pair (a, b) (reduced angle rounded to fp32: 2^-24 pi; sincosf and
the products: a few fp32 ulps).  fp32 outputs must lie within eps of the oracle; bf16 outputs,
rounded once, within 2^-8 |ref| + 2 eps.  V rows, components past rotary_dim and every cache row
that is not a tree slot are bit-exact.
"""
import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import rope as OR
from oracle import tree as OT
from speculative_decoding_draft_tree_gb300 import binding as B
from speculative_decoding_draft_tree_gb300 import workloads as W
from speculative_decoding_draft_tree_gb300.api import VerifyStep

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _pair_scale(x, rotary_dim, interleaved):
    """|a| + |b| of the pair each component belongs to (the error scale), 0 past rotary_dim."""
    s = np.zeros_like(x)
    for ia, ib in OR.pair_indices(rotary_dim, interleaved):
        m = np.abs(x[..., ia]) + np.abs(x[..., ib])
        s[..., ia] = m
        s[..., ib] = m
    return s


def _assert_rotated(got, ref, x_in, dtype, rotary_dim, interleaved):
    eps = 1e-6 * _pair_scale(x_in, rotary_dim, interleaved)
    tol = eps if dtype == "f32" else 2.0 ** -8 * np.abs(ref) + 2 * eps
    bad = np.abs(got - ref) > tol
    assert not bad.any(), (int(bad.sum()), float(np.abs(got - ref).max()))
    # pass-through components are copied exactly
    np.testing.assert_array_equal(got[..., rotary_dim:], ref[..., rotary_dim:])


def _tree_rows(w, table, prefix, no):
    """(request, node, physical block, row) of every tree slot, from the block table."""
    out = []
    for r in range(w.B):
        for i in range(no[r + 1] - no[r]):
            s = prefix[r] + i
            out.append((r, no[r] + i, int(table[r, s // w.bs]), s % w.bs))
    return out


def _run(w, rotary_dim, interleaved, base, in_place=False, corrupt=None, fused=False):
    step = VerifyStep(w)
    if corrupt is not None:
        corrupt(w)
    if not fused:
        step.tree_build()
    q_raw = w.q.clone()
    k_new, v_new = W.new_tree_kv(w)
    kc0, vc0 = step.k_layer0.clone(), step.v_layer0.clone()
    q_out = q_raw if in_place else torch.full_like(q_raw, 7.0)
    p = B.rope_params(q_raw, q_out, k_new, v_new, step.k_layer0, step.v_layer0, w.block_table,
                      w.prefix_len, w.node_offset, step.pos_id, step.req_status, base, rotary_dim,
                      interleaved)
    if fused:
        B.spec_tree_build_rope_kv_write(w.parent, w.node_offset, w.prefix_len, w.T_max,
                                        step.depth, step.pos_id, step.anc_mask, step.is_internal,
                                        step.req_status, p)
    else:
        B.spec_tree_rope_kv_write(p)
    torch.cuda.synchronize()
    return step, q_out, (q_raw if not in_place else None), k_new, v_new, kc0, vc0


def _oracle(w, q_raw_np, k_new, v_new, kc0, vc0, rotary_dim, interleaved, base):
    no = w.node_offset.cpu().numpy()
    prefix = w.prefix_len.cpu().numpy()
    tb = OT.tree_build(w.parent.cpu().numpy(), no, prefix, w.T_max)
    return OR.tree_rope_kv_write(q_raw_np, _np(k_new), _np(v_new), tb["pos_id"], no, prefix,
                                 w.block_table.cpu().numpy(), _np(kc0), _np(vc0), base,
                                 rotary_dim, interleaved, req_status=tb["status"])


def _check_full(w, step, q_out, q_raw_np, k_new, v_new, kc0, vc0, rotary_dim, interleaved, base):
    orc = _oracle(w, q_raw_np, k_new, v_new, kc0, vc0, rotary_dim, interleaved, base)
    st = step.req_status.cpu().numpy()
    assert st.tolist() == orc["status"].tolist()
    ok = ~np.isnan(orc["q"][:, 0, 0])
    _assert_rotated(_np(q_out)[ok], orc["q"][ok], q_raw_np[ok], w.dtype, rotary_dim, interleaved)
    k_got, v_got = _np(step.k_layer0), _np(step.v_layer0)
    written = np.zeros(k_got.shape[0:1] + k_got.shape[2:3], dtype=bool)   # [blocks, rows]
    no, prefix, table = (w.node_offset.cpu().numpy(), w.prefix_len.cpu().numpy(),
                         w.block_table.cpu().numpy())
    for r, n, blk, row in _tree_rows(w, table, prefix, no):
        if orc["status"][r]:
            continue
        written[blk, row] = True
        _assert_rotated(k_got[blk, :, row], orc["k_cache"][blk, :, row], _np(k_new[n]), w.dtype,
                        rotary_dim, interleaved)
    np.testing.assert_array_equal(v_got, orc["v_cache"])
    keep = ~written
    np.testing.assert_array_equal(k_got.transpose(0, 2, 1, 3)[keep],
                                  _np(kc0).transpose(0, 2, 1, 3)[keep])
    return orc


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5])
def test_rope_small_configs(cid, interleaved, fused):
    w = W.make_config(cid, scale="small", device="cuda")
    step, q_out, q_raw, k_new, v_new, kc0, vc0 = _run(w, w.d, interleaved, 10000.0, fused=fused)
    _check_full(w, step, q_out, _np(q_raw), k_new, v_new, kc0, vc0, w.d, interleaved, 10000.0)
    if fused:   # the fused launch also produced the tree outputs
        import parity_util as PU
        PU.check_tree(w, step, PU.snapshot(w))


@pytest.mark.parametrize("cid", [1, 3, 5])
def test_fused_equals_two_calls(cid):
    """spec_tree_build_rope_kv_write gives bit for bit what spec_tree_build followed by
    spec_tree_rope_kv_write gives."""
    outs = []
    for fused in (False, True):
        w = W.make_config(cid, scale="small", device="cuda")
        step, q_out, _, _, _, _, _ = _run(w, w.d, False, 10000.0, fused=fused)
        outs.append([t.clone() for t in (q_out, step.k_layer0, step.v_layer0, step.depth,
                                         step.pos_id, step.anc_mask, step.is_internal,
                                         step.req_status)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


@pytest.mark.parametrize("cid,rd,base", [(1, 32, 1e6), (2, 64, 500000.0), (5, 64, 10000.0),
                                         (4, 128, 1e6)])
def test_rope_partial_rotary_and_bases(cid, rd, base):
    w = W.make_config(cid, scale="small", device="cuda")
    step, q_out, q_raw, k_new, v_new, kc0, vc0 = _run(w, rd, False, base)
    _check_full(w, step, q_out, _np(q_raw), k_new, v_new, kc0, vc0, rd, False, base)


def test_rope_in_place_matches_out_of_place():
    w = W.make_config(4, scale="small", device="cuda")
    q0 = _np(w.q)
    _, q_sep, _, _, _, _, _ = _run(w, w.d, False, 10000.0)
    w2 = W.make_config(4, scale="small", device="cuda")
    step, q_in_place, _, k_new, v_new, kc0, vc0 = _run(w2, w.d, False, 10000.0, in_place=True)
    np.testing.assert_array_equal(_np(q_in_place), _np(q_sep))
    _check_full(w2, step, q_in_place, q0, k_new, v_new, kc0, vc0, w.d, False, 10000.0)


@pytest.mark.parametrize("fused", [False, True])
def test_rope_bad_block_and_bad_tree_are_skipped(fused):
    w = W.make_config(5, scale="small", device="cuda")
    P1 = int(w.prefix_len[1])
    nb = w.k_cache.shape[1]

    def corrupt(w):
        t = w.block_table.clone()
        t[1, (P1 + 2) // w.bs] = nb + 5          # request 1: one tree slot outside the pool
        w.block_table.copy_(t)
        par = w.parent.clone()
        par[int(w.node_offset[2]) + 1] = 5       # request 2: node 1's parent is not below it
        w.parent.copy_(par)

    step, q_out, q_raw, k_new, v_new, kc0, vc0 = _run(w, w.d, False, 10000.0, corrupt=corrupt,
                                                      fused=fused)
    st = step.req_status.cpu().numpy()
    assert st[1] == B.REQ_BITS["BAD_BLOCK"] and st[2] == B.REQ_BITS["BAD_PARENT"]
    assert st[0] == 0 and st[3] == 0
    no = w.node_offset.cpu().numpy()
    # skipped requests' q_out keeps its fill
    assert (_np(q_out)[no[1]:no[3]] == 7.0).all()
    _check_full(w, step, q_out, _np(q_raw), k_new, v_new, kc0, vc0, w.d, False, 10000.0)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("cid", [2, 3, 4, 5])
def test_rope_full_size_sampled(cid, fused):
    """The full workload (launch configuration of the benchmark): every tree slot and every q
    row against the oracle's rotation; cache rows next to the tree region unchanged."""
    w = W.make_config(cid, scale="full", device="cuda")
    step = VerifyStep(w)
    q_raw = w.q.clone()
    k_new, v_new = W.new_tree_kv(w)
    step.enable_rope(q_raw, k_new, v_new, fused=fused)
    no, prefix, table = (w.node_offset.cpu().numpy(), w.prefix_len.cpu().numpy(),
                         w.block_table.cpu().numpy())
    # the block before each request's first tree slot's block holds prefix slots only
    pre = torch.as_tensor([table[r, prefix[r] // w.bs - 1] for r in range(w.B)], device="cuda")
    assert (prefix >= w.bs).all()
    before = _np(step.k_layer0[pre])
    if fused:
        step.tree_build_rope()
    else:
        step.tree_build()
        step.rope()
    torch.cuda.synchronize()
    tb = OT.tree_build(w.parent.cpu().numpy(), no, prefix, w.T_max)
    assert not tb["status"].any() and not step.req_status.cpu().numpy().any()
    pos = tb["pos_id"]
    ref_q = OR.rope(_np(q_raw), pos[:, None], 10000.0, w.d, False)
    _assert_rotated(_np(w.q), ref_q, _np(q_raw), w.dtype, w.d, False)
    rows = _tree_rows(w, table, prefix, no)
    blk = torch.as_tensor([b for _, _, b, _ in rows], device="cuda")
    row = torch.as_tensor([x for _, _, _, x in rows], device="cuda")
    k_got = _np(step.k_layer0[blk, :, row])
    v_got = _np(step.v_layer0[blk, :, row])
    nodes = np.array([n for _, n, _, _ in rows])
    ref_k = OR.rope(_np(k_new)[nodes], pos[nodes][:, None], 10000.0, w.d, False)
    _assert_rotated(k_got, ref_k, _np(k_new)[nodes], w.dtype, w.d, False)
    np.testing.assert_array_equal(v_got, _np(v_new)[nodes])
    np.testing.assert_array_equal(_np(step.k_layer0[pre]), before)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("cid", [2, 4, 5])
def test_rope_then_attention_matches_oracle_chain(cid, fused):
    """tree build -> RoPE + K/V write -> tree attention on the GPU against the same chain of
    oracle functions (sampled rows)."""
    w = W.make_config(cid, scale="small", device="cuda")
    step = VerifyStep(w)
    q_raw = w.q.clone()
    k_new, v_new = W.new_tree_kv(w)
    kc0, vc0 = _np(step.k_layer0), _np(step.v_layer0)
    step.enable_rope(q_raw, k_new, v_new, fused=fused)
    step.run()
    torch.cuda.synchronize()
    no, prefix, table = (w.node_offset.cpu().numpy(), w.prefix_len.cpu().numpy(),
                         w.block_table.cpu().numpy())
    par = w.parent.cpu().numpy()
    tb = OT.tree_build(par, no, prefix, w.T_max)
    orc = OR.tree_rope_kv_write(_np(q_raw), _np(k_new), _np(v_new), tb["pos_id"], no, prefix,
                                table, kc0, vc0)
    rng = np.random.default_rng(cid)
    rows = [(int(n), int(h)) for n, h in zip(rng.integers(0, w.N, 64), rng.integers(0, w.H_q, 64))]
    att = OA.tree_attention(orc["q"], orc["k_cache"], orc["v_cache"], table, prefix, no, par,
                            w.bs, rows=rows)
    o = _np(step.o)
    for n, h in rows:
        np.testing.assert_allclose(o[n, h], att["o"][n, h], atol=2e-2, rtol=0)
