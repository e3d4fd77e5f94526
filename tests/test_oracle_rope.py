"""Pins for oracle.rope: rotary position embedding at the tree's position ids and the tree K/V
write into paged slots.

What ties it to something other than itself:
  * RoFormer's complex form (section 3.2): pair j, read as the complex number a + i b, is
    multiplied by exp(i m theta_j) -- computed here with numpy complex arithmetic;
  * the frequencies as numbers: with base 10000 and rotary_dim 8 the pairs turn by 1, 0.1,
    0.01 and 0.001 radians per position;
  * the relative-position property <R(m) q, R(n) k> = <R(m - n) q, k> and norm preservation;
  * the half-split layout is the interleaved one after a fixed permutation of components;
  * brute force over every physical cache row for the slot write;
  * end to end: for a chain tree, tree build -> RoPE + K/V write -> tree attention equals
    library causal attention over the RoPE'd sequence (sequential decoding).
"""
import numpy as np
import torch
import torch.nn.functional as F

from oracle import attention as OA
from oracle import rope as OR
from oracle import tree as OT


def _complex_rope(x, pos, base, rotary_dim, interleaved):
    x = np.asarray(x, dtype=np.float64)
    half = rotary_dim // 2
    if interleaved:
        z = x[..., 0:rotary_dim:2] + 1j * x[..., 1:rotary_dim:2]
    else:
        z = x[..., :half] + 1j * x[..., half:rotary_dim]
    freq = np.array([base ** (-(2.0 * j) / rotary_dim) for j in range(half)])
    z = z * np.exp(1j * np.asarray(pos, dtype=np.float64)[..., None] * freq)
    out = x.copy()
    if interleaved:
        out[..., 0:rotary_dim:2], out[..., 1:rotary_dim:2] = z.real, z.imag
    else:
        out[..., :half], out[..., half:rotary_dim] = z.real, z.imag
    return out


def test_position_zero_is_identity():
    x = np.random.default_rng(0).normal(size=(3, 5, 16))
    for inter in (False, True):
        np.testing.assert_array_equal(OR.rope(x, 0, interleaved=inter), x)


def test_complex_form():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(4, 6, 32))
    pos = rng.integers(0, 40000, size=(4, 6))
    for inter in (False, True):
        for rd, base in ((32, 10000.0), (16, 500000.0), (32, 1e6)):
            np.testing.assert_allclose(OR.rope(x, pos, base, rd, inter),
                                       _complex_rope(x, pos, base, rd, inter),
                                       rtol=0, atol=1e-12)


def test_frequencies_as_numbers():
    # pair j of a unit vector turns by base ** (-2j / rotary_dim) radians per position
    want = [1.0, 0.1, 0.01, 0.001]
    for j, w in enumerate(want):
        for inter in (False, True):
            ia, ib = OR.pair_indices(8, inter)[j]
            e = np.zeros(8)
            e[ia] = 1.0
            y = OR.rope(e, 1, 10000.0, 8, inter)
            assert abs(np.arctan2(y[ib], y[ia]) - w) < 1e-14
            y = OR.rope(e, 3, 10000.0, 8, inter)
            assert abs(np.arctan2(y[ib], y[ia]) - 3 * w) < 1e-14
    # the rotation is counter-clockwise: e_a -> (cos, sin), e_b -> (-sin, cos)
    e = np.zeros(8)
    e[1] = 1.0
    y = OR.rope(e, 1, 10000.0, 8, True)
    np.testing.assert_allclose(y[:2], [-np.sin(1.0), np.cos(1.0)], atol=1e-15)


def test_relative_position_and_norm():
    rng = np.random.default_rng(2)
    q, k = rng.normal(size=64), rng.normal(size=64)
    for inter in (False, True):
        for m, n in ((5, 3), (3, 5), (4096, 4090), (32768, 1), (77, 77)):
            lhs = OR.rope(q, m, 10000.0, 64, inter) @ OR.rope(k, n, 10000.0, 64, inter)
            rhs = OR.rope(q, m - n, 10000.0, 64, inter) @ k
            assert abs(lhs - rhs) < 1e-10
        y = OR.rope(q, 12345, 10000.0, 64, inter)
        assert abs(np.linalg.norm(y) - np.linalg.norm(q)) < 1e-12


def test_half_split_is_permuted_interleaved():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(7, 24))
    pos = rng.integers(0, 5000, size=7)
    perm = np.ravel(np.column_stack([np.arange(12), np.arange(12, 24)]))  # 0,12,1,13,...
    a = OR.rope(x, pos, 10000.0, 24, interleaved=False)
    b = OR.rope(x[:, perm], pos, 10000.0, 24, interleaved=True)
    np.testing.assert_allclose(a[:, perm], b, atol=1e-13)


def test_partial_rotary_leaves_tail():
    rng = np.random.default_rng(4)
    x = rng.normal(size=(5, 32))
    y = OR.rope(x, 999, 10000.0, 16, False)
    np.testing.assert_array_equal(y[:, 16:], x[:, 16:])
    np.testing.assert_allclose(y[:, :16], _complex_rope(x[:, :16], 999, 10000.0, 16, False),
                               atol=1e-12)


def _paged_case(sizes, prefix, H_q=4, H_kv=2, d=16, bs=4, seed=5):
    rng = np.random.default_rng(seed)
    B = len(sizes)
    no = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    need = [-(-(prefix[r] + sizes[r]) // bs) for r in range(B)]
    nb = sum(need) + 3
    perm = rng.permutation(nb)
    table = np.full((B, max(need) + 1), -1)
    at = 0
    for r in range(B):
        table[r, :need[r]] = perm[at:at + need[r]]
        at += need[r]
    N = int(no[-1])
    return dict(rng=rng, no=no, table=table, nb=nb, N=N, H_q=H_q, H_kv=H_kv, d=d, bs=bs,
                P=np.asarray(prefix), q=rng.normal(size=(N, H_q, d)),
                k_new=rng.normal(size=(N, H_kv, d)), v_new=rng.normal(size=(N, H_kv, d)),
                kc=rng.normal(size=(nb, H_kv, bs, d)), vc=rng.normal(size=(nb, H_kv, bs, d)))


def test_slot_write_brute_force():
    c = _paged_case([5, 1, 9], [6, 0, 13])
    pos = c["rng"].integers(0, 100, size=c["N"])
    out = OR.tree_rope_kv_write(c["q"], c["k_new"], c["v_new"], pos, c["no"], c["P"], c["table"],
                                c["kc"], c["vc"], 10000.0, 16, False)
    assert not out["status"].any()
    owner = {}
    for r in range(len(c["P"])):
        for lb, blk in enumerate(c["table"][r]):
            if blk >= 0:
                owner[int(blk)] = (r, lb)
    for blk in range(c["nb"]):
        for row in range(c["bs"]):
            want_k, want_v = c["kc"][blk, :, row], c["vc"][blk, :, row]
            if blk in owner:
                r, lb = owner[blk]
                i = lb * c["bs"] + row - c["P"][r]
                if 0 <= i < c["no"][r + 1] - c["no"][r]:
                    n = c["no"][r] + i
                    want_k = _complex_rope(c["k_new"][n], pos[n], 10000.0, 16, False)
                    want_v = c["v_new"][n]
            np.testing.assert_allclose(out["k_cache"][blk, :, row], want_k, atol=1e-12)
            np.testing.assert_array_equal(out["v_cache"][blk, :, row], want_v)
    np.testing.assert_allclose(out["q"], _complex_rope(c["q"], pos[:, None], 10000.0, 16, False),
                               atol=1e-12)


def test_bad_block_and_bad_request_are_skipped():
    c = _paged_case([4, 4], [3, 3])
    c["table"][1, 1] = c["nb"] + 7   # request 1's tree slots 4..6 fall in a bad block
    pos = np.arange(c["N"])
    out = OR.tree_rope_kv_write(c["q"], c["k_new"], c["v_new"], pos, c["no"], c["P"], c["table"],
                                c["kc"], c["vc"], req_status=[0, 0])
    assert list(out["status"]) == [0, OR.BAD_BLOCK]
    assert np.isnan(out["q"][4:]).all() and not np.isnan(out["q"][:4]).any()
    blk0 = c["table"][1, 0]
    np.testing.assert_array_equal(out["k_cache"][blk0], c["kc"][blk0])   # slot 3 not written
    out = OR.tree_rope_kv_write(c["q"], c["k_new"], c["v_new"], pos, c["no"], c["P"], c["table"],
                                c["kc"], c["vc"], req_status=[2, 0])
    assert list(out["status"]) == [2, OR.BAD_BLOCK]
    np.testing.assert_array_equal(out["k_cache"], c["kc"])
    # a negative prefix length has no cache slots: nothing of that request is written
    out = OR.tree_rope_kv_write(c["q"], c["k_new"], c["v_new"], pos, c["no"], [-1, 3], c["table"],
                                c["kc"], c["vc"], req_status=[0, 0])
    assert np.isnan(out["q"][:4]).all()
    np.testing.assert_array_equal(out["k_cache"], c["kc"])
    # a node with a negative position id is skipped: its q stays NaN and its slot unwritten
    c = _paged_case([3], [5])
    pos = np.array([5, -1, 6])
    out = OR.tree_rope_kv_write(c["q"], c["k_new"], c["v_new"], pos, c["no"], c["P"], c["table"],
                                c["kc"], c["vc"])
    assert np.isnan(out["q"][1]).all() and not np.isnan(out["q"][[0, 2]]).any()
    blk, row = c["table"][0, 6 // c["bs"]], 6 % c["bs"]   # node 1's slot: prefix 5 + 1
    np.testing.assert_array_equal(out["k_cache"][blk, :, row], c["kc"][blk, :, row])
    np.testing.assert_array_equal(out["v_cache"][blk, :, row], c["vc"][blk, :, row])


def test_chain_equals_causal_decoding():
    """A chain tree after tree build -> RoPE + K/V write -> tree attention is ordinary causal
    attention over the RoPE'd sequence of prefix + chain (sequential decoding)."""
    T, P, H, d, bs, base = 6, 10, 2, 16, 4, 10000.0
    c = _paged_case([T], [P], H_q=H, H_kv=H, d=d, bs=bs, seed=9)
    raw_k = c["rng"].normal(size=(P + T, H, d))
    raw_v = c["rng"].normal(size=(P + T, H, d))
    kc, vc = c["kc"].copy(), c["vc"].copy()
    for s in range(P):   # the prefix was cached at its own positions
        blk, row = c["table"][0, s // bs], s % bs
        kc[blk, :, row] = _complex_rope(raw_k[s], s, base, d, False)
        vc[blk, :, row] = raw_v[s]
    parent = np.arange(T) - 1
    tb = OT.tree_build(parent, c["no"], [P], T)
    out = OR.tree_rope_kv_write(c["q"], raw_k[P:], raw_v[P:], tb["pos_id"], c["no"], [P],
                                c["table"], kc, vc, base)
    att = OA.tree_attention(out["q"], out["k_cache"], out["v_cache"], c["table"], [P], c["no"],
                            parent, bs)
    qs = torch.tensor(_complex_rope(c["q"], P + np.arange(T)[:, None], base, d, False))
    ks = torch.tensor(_complex_rope(raw_k, np.arange(P + T)[:, None], base, d, False))
    vs = torch.tensor(raw_v)
    for h in range(H):
        qh = torch.cat([torch.zeros(P, d, dtype=torch.float64), qs[:, h]]).view(1, 1, P + T, d)
        ref = F.scaled_dot_product_attention(qh, ks[:, h].view(1, 1, P + T, d),
                                             vs[:, h].view(1, 1, P + T, d), is_causal=True)
        np.testing.assert_allclose(att["o"][:, h], ref.view(P + T, d)[P:].numpy(), atol=1e-12)
