"""GPU <-> oracle parity through the C-ABI (spec_tree_build, spec_tree_attention, spec_verify,
spec_kv_compact) on the five workloads at oracle-friendly sizes, the edge cases, injected data
errors and guard bands."""
import numpy as np
import pytest
import torch

import parity_util as PU
from speculative_decoding_draft_tree_gb300 import binding as B
from speculative_decoding_draft_tree_gb300 import workloads as W
from speculative_decoding_draft_tree_gb300.api import VerifyStep

pytestmark = pytest.mark.gpu


def _sync():
    torch.cuda.synchronize()


def run_and_check(w, rule=B.SPEC_SIBLING_RESIDUAL, attention=True, rows=None):
    snap = PU.snapshot(w)
    step = VerifyStep(w, sibling_rule=rule)
    step.tree_build()
    _sync()
    PU.check_tree(w, step, snap)
    if attention:
        step.attention()
        _sync()
        PU.check_attention(w, step, snap, rows)
    step.verify()
    _sync()
    orc = PU.oracle_verify(w, snap, rule)
    draws, exempt = PU.check_verify(w, step, orc)
    kb = PU.cache_region(w.k_cache, w, snap, range(w.B))
    vb = PU.cache_region(w.v_cache, w, snap, range(w.B))
    step.compact()
    _sync()
    PU.check_compact(w, step, snap, kb, vb)
    return step, orc, draws, exempt


@pytest.mark.parametrize("tau", [1.0, 0.0])
@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5])
def test_verify_small_configs(cid, tau):
    w = W.make_config(cid, scale="small", device="cuda", tau=tau, num_layers=2)
    run_and_check(w, attention=False)


@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5])
def test_attention_small_configs(cid):
    w = W.make_config(cid, scale="small", device="cuda")
    run_and_check(w, attention=True)


@pytest.mark.parametrize("sigma", [0.5, 2.0])
def test_chain_noise_sweep(sigma):
    w = W.make_config(2, scale="small", device="cuda", sigma=sigma)
    run_and_check(w, attention=False)


@pytest.mark.parametrize("cid", [3, 4, 5])
def test_independent_sibling_rule(cid):
    w = W.make_config(cid, scale="small", device="cuda")
    run_and_check(w, rule=B.SPEC_SIBLING_INDEPENDENT, attention=False)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_draft_probabilities(dtype):
    w = W.chain_workload(B=5, gamma=4, V=2003, dtype=dtype, H_q=4, H_kv=4,
                         d=64 if dtype == "f32" else 128, prefix=40, tau=1.0, target_std=2.0,
                         noise_std=1.0, device="cuda", draft_kind=W.DRAFT_PROBS)
    run_and_check(w, attention=False)


@pytest.mark.parametrize("tau", [0.7, 1.6])
def test_other_temperatures(tau):
    w = W.make_config(4, scale="small", device="cuda", tau=tau)
    run_and_check(w, attention=False)


@pytest.mark.parametrize("P", [0, 15, 16, 17, 31])
def test_single_token_trees_and_block_boundaries(P):
    # T = 1 (plain decode), prefix lengths at block boundaries, odd vocabulary
    w = W.chain_workload(B=3, gamma=0, V=1001, dtype="bf16", H_q=8, H_kv=2, d=128, prefix=P,
                         tau=1.0, target_std=3.0, noise_std=1.0, device="cuda", T_max=4)
    run_and_check(w, attention=True)


def test_chain_block_boundaries_f32():
    w = W.chain_workload(B=4, gamma=5, V=999, dtype="f32", H_q=4, H_kv=2, d=64,
                         prefix=[0, 15, 16, 33], tau=1.0, target_std=2.0, noise_std=1.0,
                         device="cuda")
    run_and_check(w, attention=True)


def test_maximum_tree_size():
    # trees of exactly SPEC_MAX_TREE = 256 nodes (Medusa ks = (15, 16): 1 + 15 + 240), eight
    # query heads per KV head: 2048 query rows per request, 16 M-tiles
    w = W.medusa_workload(B=2, ks=(15, 16), V=3001, dtype="bf16", H_q=8, H_kv=1, d=128,
                          prefix=[40, 77], tau=1.0, device="cuda")
    assert w.tree_sizes() == [256, 256]
    run_and_check(w, attention=True)


def _corrupt_workload():
    w = W.make_config(5, scale="small", device="cuda", num_layers=2)
    no = w.node_offset.cpu().numpy()
    par = w.parent.clone()
    par[no[0] + 3] = 3                       # request 0: parent[i] == i
    w.parent.copy_(par)
    w.tokens[no[1] + 2] = w.V                # request 1: token id >= V
    # request 2: an internal node whose draft row is out of range
    internal_local = int(torch.nonzero(w.draft_row[no[2]:no[3]] >= 0)[1])
    w.draft_row[no[2] + internal_local] = w.R + 7
    # request 3: a block-table entry of the tree region out of range
    P3 = int(w.prefix_len[3])
    w.block_table[3, P3 // w.bs] = w.k_cache.shape[1] + 5
    return w


def test_injected_data_errors():
    w = _corrupt_workload()
    snap = PU.snapshot(w)
    step = VerifyStep(w)
    step.run()
    _sync()
    st = PU.np_(step.req_status)
    assert st[0] & B.REQ_BITS["BAD_PARENT"]
    assert st[1] & B.REQ_BITS["BAD_TOKEN"]
    assert st[2] & B.REQ_BITS["BAD_DRAFT_ROW"]
    assert st[3] & B.REQ_BITS["BAD_BLOCK"]
    assert (PU.np_(step.out_len)[:3] == 0).all()
    assert (PU.np_(step.n_acc)[:3] == -1).all()
    # the rolled-back requests keep their prefix length
    assert PU.np_(step.new_kv_len)[:3].tolist() == snap["prefix_len"][:3].tolist()
    # the library is still usable afterwards
    w2 = W.make_config(5, scale="small", device="cuda")
    run_and_check(w2, attention=False)


def test_oversize_tree_flagged():
    w = W.make_config(5, scale="small", device="cuda")
    sizes = w.tree_sizes()
    w.T_max = 40
    w.max_path = 40
    step = VerifyStep(w)
    step.tree_build()
    step.verify()
    _sync()
    st = PU.np_(step.req_status)
    for r, T in enumerate(sizes):
        assert bool(st[r] & B.REQ_BITS["BAD_SIZE"]) == (T > 40)


def test_host_validation_errors():
    w = W.make_config(2, scale="small", device="cuda")
    step = VerifyStep(w)
    bad = B.verify_params(w.target, w.draft, w.draft_kind, w.draft_row, w.tokens, w.parent,
                          w.node_offset, step.depth, step.is_internal, w.uniforms, -1.0, w.V,
                          w.T_max, w.max_path, step.req_status, step.out_tokens, step.out_len,
                          step.path, step.n_acc)
    with pytest.raises(B.SpecError, match="INVALID_ARG"):
        B.spec_verify(bad, step.ver_ws)
    with pytest.raises(B.SpecError, match="INVALID_ARG"):
        B.spec_verify(step.ver, step.ver_ws[:16])   # workspace too small
    p = B.attention_params(w.q, step.k_layer0, step.v_layer0, w.block_table, w.prefix_len,
                           w.node_offset, step.anc_mask, w.T_max, step.o, None, step.req_status)
    p.q = p.q + 2                                       # misaligned
    with pytest.raises(B.SpecError, match="INVALID_ARG"):
        B.spec_tree_attention(p, step.attn_ws)
    with pytest.raises(B.SpecError, match="INVALID_ARG"):
        B.spec_tree_build(w.parent, w.node_offset, w.prefix_len, 300, step.depth, step.pos_id,
                          step.anc_mask, step.is_internal, step.req_status)


def test_guard_bands_untouched():
    w = W.make_config(4, scale="small", device="cuda")
    step = VerifyStep(w)
    pad = 1024
    sentinel = -777
    big = {}
    for name in ("out_tokens", "path", "out_len", "n_acc", "rejections", "new_kv_len",
                 "blocks_in_use", "slot_map", "depth", "pos_id"):
        t = getattr(step, name)
        buf = torch.full((t.numel() + 2 * pad,), sentinel, dtype=t.dtype, device=t.device)
        view = buf[pad:pad + t.numel()].view(t.shape)
        big[name] = buf
        setattr(step, name, view)
    # rebuild parameter blocks over the guarded views
    step.ver = B.verify_params(w.target, w.draft, w.draft_kind, w.draft_row, w.tokens, w.parent,
                               w.node_offset, step.depth, step.is_internal, w.uniforms, w.tau,
                               w.V, w.T_max, w.max_path, step.req_status, step.out_tokens,
                               step.out_len, step.path, step.n_acc, step.rejections)
    step.comp = B.compact_params(w.k_cache, w.v_cache, w.block_table, w.prefix_len, step.path,
                                 step.n_acc, step.req_status, step.new_kv_len, step.slot_map,
                                 step.blocks_in_use, w.max_path)
    step.tree_build()
    step.verify()
    step.compact()
    _sync()
    for name, buf in big.items():
        assert (buf[:pad] == sentinel).all() and (buf[-pad:] == sentinel).all(), name


def test_twin_and_host_round_trip():
    # a twin step (own input copies, shared KV cache) fed the same host inputs gives the same
    # round as the original, whether run through run_from_host or upload / run / download
    w = W.make_config(2, scale="small", device="cuda", num_layers=2)
    step = VerifyStep(w)
    host_in = step.pinned_host_inputs()
    k0 = w.k_cache.clone()
    v0 = w.v_cache.clone()
    out_a = step.host_output_buffers()
    step.run_from_host(host_in, out_a)
    _sync()
    res_a = {k: step.results()[k].cpu().clone() for k in ("out_tokens", "out_len", "path", "n_acc")}
    w.k_cache.copy_(k0)
    w.v_cache.copy_(v0)
    twin = step.twin()
    assert twin.w.k_cache.data_ptr() == w.k_cache.data_ptr()
    assert twin.w.target.data_ptr() != w.target.data_ptr()
    out_b = twin.host_output_buffers()
    copy_stream = torch.cuda.Stream()
    packed_in = twin.pinned_host_inputs()
    assert set(packed_in) == {"_pack"}
    twin.upload(packed_in, copy_stream)
    torch.cuda.current_stream().wait_stream(copy_stream)
    twin.run()
    twin.download(out_b)
    _sync()
    for k, v in res_a.items():
        assert torch.equal(twin.results()[k].cpu(), v), k
    for k in ("out_tokens", "out_len", "new_kv_len"):
        assert torch.equal(out_a[k], out_b[k]), k


def test_graph_replay_matches_stream_launches():
    """A round captured as a CUDA graph (programmatic dependencies inside) gives the same results
    as the same round launched on a stream."""
    warm = VerifyStep(W.make_config(4, scale="small", device="cuda", num_layers=2))
    warm.run()   # first calls set per-device kernel attributes, which capture does not allow
    torch.cuda.synchronize()
    outs = []
    for use_graph in (False, True):
        w = W.make_config(4, scale="small", device="cuda", num_layers=2)
        step = VerifyStep(w)
        if use_graph:
            g = step.capture_graph()
            g.replay()
        else:
            step.run()
        torch.cuda.synchronize()
        out = {k: v.clone() for k, v in step.results().items() if v is not None}
        out["k_cache"] = w.k_cache.clone()
        outs.append(out)
    for k in outs[0]:
        assert torch.equal(outs[0][k], outs[1][k]), k


@pytest.mark.parametrize("B_req,prefix,contiguous", [(3, 300, True), (1, 5000, False), (5, 40, False)])
def test_attention_graph_replays_merge_cut_units(B_req, prefix, contiguous):
    """Units cut across CTA ranges are merged by log-sum-exp from partial pieces kept in the
    workspace, which is filled with stale bytes first (its contents need not be initialised).
    Chains at these sizes cut units into 2 pieces (prefix 300), up to ~11 pieces (prefix 5000)
    and cut none (prefix 40); every launch -- the stream launch and three replays of a captured
    graph, the outputs cleared before each -- must give the oracle's result, bit-identical across
    launches."""
    w = W.chain_workload(B=B_req, gamma=5, V=1009, dtype="bf16", H_q=4, H_kv=4, d=128,
                         prefix=prefix, tau=1.0, target_std=2.0, noise_std=1.0, device="cuda",
                         contiguous=contiguous)
    snap = PU.snapshot(w)
    step = VerifyStep(w)
    step.attn_ws.fill_(0xA5)   # counters and partials as stale bytes
    step.tree_build()
    step.attention()
    _sync()
    PU.check_attention(w, step, snap)
    want_o, want_lse = step.o.clone(), step.lse.clone()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            step.attention(side)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        step.o.zero_()
        step.lse.fill_(float("nan"))
        g.replay()
        _sync()
        assert torch.equal(step.o, want_o)
        assert torch.equal(step.lse, want_lse)


def test_round_pipeline_alternating_inputs():
    # rounds of two different batches (same shape) submitted alternately through the
    # double-buffered pipeline land in the right host buffers with the results that each batch
    # gives when run alone
    from speculative_decoding_draft_tree_gb300.api import RoundPipeline
    wa = W.make_config(2, scale="small", device="cuda", num_layers=2)
    wb = W.make_config(2, scale="small", device="cuda", num_layers=2,
                       seeds=dict(logits=11, drafting=12, qkv=13))
    keys = ("out_tokens", "out_len", "new_kv_len")
    want = []
    for w in (wa, wb):
        s = VerifyStep(w)
        s.run()
        _sync()
        want.append({k: getattr(s, k).cpu().clone() for k in keys})
    assert not torch.equal(want[0]["out_tokens"], want[1]["out_tokens"])
    pipe = RoundPipeline(VerifyStep(wa))
    host = [pipe.pinned_host_inputs(), VerifyStep(wb).twin().pinned_host_inputs()]
    for n_rounds in (2, 5):
        first = pipe.count
        for i in range(n_rounds):
            pipe.submit(host[i % 2])
        pipe.finish()
        _sync()
        for i in (n_rounds - 2, n_rounds - 1):
            got = pipe.host_outputs(first + i)
            for k in keys:
                assert torch.equal(got[k], want[i % 2][k]), (n_rounds, i, k)
