"""The parity harness's own bars, on the CPU, with stand-ins for the GPU's outputs built from the
oracle's results: check_verify passes the oracle's own results, fails a divergence whose
decisions all lie clear of the fp32 band, and exempts one (and counts it) only when the oracle's
decision at the divergence lies within the band; check_attention passes the oracle's output in
the kernel's dtype and fails an output or LSE element beyond its bar; check_tree fails a single
flipped mask bit; check_compact fails one wrong element of a moved row and a wrong block count;
the draft-tree comparison's near-tie detector flags a near tie at a top-K boundary and neither
an exact tie nor a clear row; the RoPE bar passes the oracle rounded once to fp32 or bf16 and
fails the opposite rotation and a changed pass-through component."""
import copy
import types

import numpy as np
import pytest
import torch

import parity_util as PU
from speculative_decoding_draft_tree_gb300 import workloads as W


@pytest.fixture(autouse=True)
def keep_tally():
    # the suite-wide exemption tally belongs to the GPU parity tests
    saved = dict(PU.TALLY)
    yield
    PU.TALLY.clear()
    PU.TALLY.update(saved)


def _case():
    w = W.make_config(3, scale="small", device="cpu")   # Medusa (3, 5, 7), two requests
    orc = PU.oracle_verify(w, PU.snapshot(w))
    assert not orc["status"].any()
    return w, orc


def _as_step(w, orc):
    path = np.full((w.B, w.max_path), -1, dtype=np.int32)
    toks = np.full((w.B, w.max_path), -1, dtype=np.int32)
    for r in range(w.B):
        path[r, :len(orc["path"][r])] = orc["path"][r]
        toks[r, :len(orc["out_tokens"][r])] = orc["out_tokens"][r]
    t = torch.from_numpy
    return types.SimpleNamespace(
        req_status=t(orc["status"].astype(np.int32)), out_len=t(orc["out_len"].astype(np.int32)),
        n_acc=t(orc["n_acc"].astype(np.int32)), path=t(path), out_tokens=t(toks),
        rejections=t(orc["rejections"].astype(np.int32)))


def test_the_oracles_own_results_pass():
    w, orc = _case()
    draws, exempt = PU.check_verify(w, _as_step(w, orc), orc)
    assert draws >= w.B and exempt == 0


def test_a_divergence_clear_of_the_band_fails():
    w, orc = _case()
    assert not any(PU._near(orc["events"][0], n) for n in orc["path"][0])
    step = _as_step(w, orc)
    L = int(orc["out_len"][0])
    step.out_tokens[0, L - 1] = (int(step.out_tokens[0, L - 1]) + 1) % w.V   # another final token
    with pytest.raises(AssertionError):
        PU.check_verify(w, step, orc)
    step = _as_step(w, orc)                       # a path one node shorter
    if L >= 2:
        step.path[0, L - 1] = -1
        step.n_acc[0] -= 1
        step.out_len[0] -= 1
        with pytest.raises(AssertionError):
            PU.check_verify(w, step, orc)
    step = _as_step(w, orc)                       # a status bit the oracle did not set
    step.req_status[1] = 4
    with pytest.raises(AssertionError):
        PU.check_verify(w, step, orc)


def test_a_divergence_within_the_band_is_exempted_and_counted():
    w, orc = _case()
    stop = orc["path"][0][-1]
    near = copy.deepcopy(orc)
    # the oracle's final draw at the stop node put within the band of a CDF edge
    near["events"][0] = [e if not (e[0] == "sample" and e[1] == stop)
                         else (e[0], e[1], e[2], 0.5 * PU.BAND) for e in orc["events"][0]]
    assert PU._near(near["events"][0], stop)
    step = _as_step(w, orc)
    L = int(orc["out_len"][0])
    step.out_tokens[0, L - 1] = (int(step.out_tokens[0, L - 1]) + 1) % w.V
    before = PU.TALLY["exempt"]
    draws, exempt = PU.check_verify(w, step, near)
    assert exempt == 1 and PU.TALLY["exempt"] == before + 1
    # the same divergence in the other request, whose decisions are clear of the band, fails
    step.out_tokens[1, int(orc["out_len"][1]) - 1] += 1
    with pytest.raises(AssertionError):
        PU.check_verify(w, step, near)


@pytest.mark.parametrize("cid", [1, 3])     # fp32 chain, bf16 Medusa tree
def test_the_attention_bar(cid):
    from oracle import attention as OA
    w = W.make_config(cid, scale="small", device="cpu")
    snap = PU.snapshot(w)
    orc = OA.tree_attention(PU.f32(w.q).astype(np.float64), w.k_cache[0].float().numpy(),
                            w.v_cache[0].float().numpy(), snap["block_table"], snap["prefix_len"],
                            snap["node_offset"], snap["parent"], w.bs)
    td = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    step = types.SimpleNamespace(req_status=torch.zeros(w.B, dtype=torch.int32),
                                 o=torch.from_numpy(orc["o"]).to(td),
                                 lse=torch.from_numpy(orc["lse"]).float())
    assert PU.check_attention(w, step, snap) < (2e-2 if w.dtype == "bf16" else 1e-5)
    # one output element off by more than the bar (bf16: 2e-2 absolute; fp32: 1e-5 relative)
    bad = step.o.clone()
    bad[1, 0, 3] += 0.05 if w.dtype == "bf16" else 1e-3 * (1 + abs(float(bad[1, 0, 3])))
    with pytest.raises(AssertionError):
        PU.check_attention(w, types.SimpleNamespace(req_status=step.req_status, o=bad,
                                                    lse=step.lse), snap)
    bad_lse = step.lse.clone()
    bad_lse[2, 1] += 1e-3
    with pytest.raises(AssertionError):
        PU.check_attention(w, types.SimpleNamespace(req_status=step.req_status, o=step.o,
                                                    lse=bad_lse), snap)


def test_the_tree_bar():
    from oracle import tree as OT
    w = W.make_config(4, scale="small", device="cpu")   # SpecInfer trees
    snap = PU.snapshot(w)
    orc = OT.tree_build(snap["parent"], snap["node_offset"], snap["prefix_len"], w.T_max)
    words = np.zeros((w.N, (w.T_max + 31) // 32), dtype=np.uint32)
    no = snap["node_offset"]
    for r in range(w.B):
        o, T = int(no[r]), int(no[r + 1] - no[r])
        for i, j in zip(*np.nonzero(orc["mask"][r])):
            words[o + i, j >> 5] |= np.uint32(1) << np.uint32(j & 31)
    t = torch.from_numpy

    def step(anc):
        return types.SimpleNamespace(
            req_status=torch.zeros(w.B, dtype=torch.int32), depth=t(orc["depth"].astype(np.int32)),
            pos_id=t(orc["pos_id"].astype(np.int32)),
            is_internal=t(orc["is_internal"].astype(np.uint8)), anc_mask=t(anc.view(np.int32)))

    PU.check_tree(w, step(words), snap)
    bad = words.copy()
    bad[int(no[1]) + 2, 0] ^= np.uint32(1)    # node 2 of request 1 loses its root bit
    with pytest.raises(AssertionError):
        PU.check_tree(w, step(bad), snap)


def test_the_compaction_bar():
    from oracle import compact as OC
    w = W.make_config(3, scale="small", device="cpu", num_layers=2)
    snap = PU.snapshot(w)
    orc = PU.oracle_verify(w, snap)
    kb = PU.cache_region(w.k_cache, w, snap, range(w.B))
    vb = PU.cache_region(w.v_cache, w, snap, range(w.B))
    comp = OC.kv_compact(w.k_cache.float().numpy(), w.v_cache.float().numpy(), snap["block_table"],
                         snap["prefix_len"], orc["path"], orc["n_acc"], w.bs, w.max_path,
                         status=orc["status"])
    assert (comp["slot_map"][..., 0] != comp["slot_map"][..., 1]).any()   # rows do move
    w.k_cache.copy_(torch.from_numpy(comp["k"]).to(w.k_cache.dtype))      # exact: bf16 values
    w.v_cache.copy_(torch.from_numpy(comp["v"]).to(w.v_cache.dtype))
    step = _as_step(w, orc)
    t = torch.from_numpy
    step.new_kv_len = t(comp["new_kv_len"].astype(np.int32))
    step.slot_map = t(comp["slot_map"].astype(np.int32))
    step.blocks_in_use = t(comp["blocks_in_use"].astype(np.int32))
    PU.check_compact(w, step, snap, kb, vb)
    # one element of a moved row written wrong
    r, d = next((r, d) for r in range(w.B) for d in range(w.max_path)
                if comp["slot_map"][r, d, 0] != comp["slot_map"][r, d, 1])
    dst = int(comp["slot_map"][r, d, 1])
    blk = int(snap["block_table"][r, dst // w.bs])
    keep = w.v_cache[1, blk, 0, dst % w.bs, 5].clone()
    w.v_cache[1, blk, 0, dst % w.bs, 5] += 1.0
    with pytest.raises(AssertionError):
        PU.check_compact(w, step, snap, kb, vb)
    w.v_cache[1, blk, 0, dst % w.bs, 5] = keep
    PU.check_compact(w, step, snap, kb, vb)
    step.blocks_in_use[r] += 1
    with pytest.raises(AssertionError):
        PU.check_compact(w, step, snap, kb, vb)


def test_the_draft_tree_near_tie_detector():
    # the draft-tree comparison exempts only requests that pass a decision fp32 cannot settle
    import test_gpu_draft_tree as TG
    from oracle import draft_tree as OD
    K, V = 2, 6
    clear = np.array([3.0, 1.0, 0.0, -1.0, -2.0, -3.0])      # top-2 and the 3rd well apart
    near = np.array([3.0, 1.0, 1.0 - 1e-6, -1.0, -2.0, -3.0])  # 2nd and 3rd within fp32's reach
    exact = np.array([3.0, 1.0, 1.0, -1.0, -2.0, -3.0])       # an exact tie: lower id both sides
    rows_np = [np.stack([clear, clear, near, near, exact, exact])]   # level 1: rows r * K + j
    log = {}

    def rows_of_level(level, chosen):
        log[level] = [list(c) for c in chosen]
        return ([[r * K + j for j in range(len(chosen[r]))] for r in range(3)],
                [[rows_np[0][r * K + j] for j in range(len(chosen[r]))] for r in range(3)])

    pool, kept, packed = OD.build([0, 0, 0], rows_of_level, K, 1, 10 ** 6)
    assert TG._near_ties(pool, log, rows_np, K, 1.0, 10 ** 6) == {1}


def test_the_rope_bar():
    import test_gpu_rope as TGR
    from oracle import rope as OR
    g = torch.Generator().manual_seed(3)
    x = torch.randn((6, 4, 128), generator=g).bfloat16().double().numpy()   # exact in bf16
    for inter in (False, True):
        ref = OR.rope(x, 1000, 10000.0, 64, inter)
        # the oracle's value rounded once to the output type passes
        TGR._assert_rotated(ref.astype(np.float32).astype(np.float64), ref, x, "f32", 64, inter)
        TGR._assert_rotated(torch.from_numpy(ref).bfloat16().double().numpy(), ref, x, "bf16",
                            64, inter)
        # the rotation the other way fails, in either output type
        wrong = OR.rope(x, -1000, 10000.0, 64, inter)
        for dt in ("f32", "bf16"):
            with pytest.raises(AssertionError):
                TGR._assert_rotated(wrong, ref, x, dt, 64, inter)
        # a component past rotary_dim must be copied exactly
        tail = ref.copy()
        tail[0, 0, 100] += 1e-3
        with pytest.raises(AssertionError):
            TGR._assert_rotated(tail, ref, x, "f32", 64, inter)
