"""spec_verify's forms against the oracle: the one-launch cluster form (trees of at most 32
nodes whose row slices fit a CTA), the two-launch form (row statistics kernel + walk kernel) and
the walk alone forming the statistics of the nodes it visits, chosen per call by the verify_path
field, on chains and small trees (sibling residual and independent
rules), draft logits and probabilities, tau = 0, ragged vocabularies, data errors and more
requests than one wave of clusters."""
import numpy as np
import pytest
import torch

import parity_util as PU
from speculative_decoding_draft_tree_gb300 import binding as B
from speculative_decoding_draft_tree_gb300 import workloads as W
from speculative_decoding_draft_tree_gb300.api import VerifyStep

pytestmark = pytest.mark.gpu

PATHS = {"cluster": B.SPEC_VERIFY_PATH_AUTO, "split": B.SPEC_VERIFY_PATH_SPLIT,
         "walk": B.SPEC_VERIFY_PATH_WALK}


@pytest.fixture(params=sorted(PATHS))
def path(request):
    return request.param


def _medusa(V=3001, dtype="bf16", tau=1.0, B_=4, ks=(2, 3, 2)):
    return W.medusa_workload(B=B_, ks=ks, V=V, dtype=dtype, H_q=4, H_kv=4, d=128, prefix=40,
                             tau=tau, device="cuda")


def _specinfer(V=2001, dtype="f32", tau=0.7, B_=4, schedule=(3, 2, 1)):
    return W.specinfer_workload(B=B_, schedule=schedule, V=V, dtype=dtype, H_q=4, H_kv=4, d=64,
                                prefix=40, tau=tau, device="cuda")


WORKLOADS = {
    "chain_bf16": lambda: W.make_config(2, scale="small", device="cuda"),
    "chain_greedy": lambda: W.make_config(2, scale="small", device="cuda", tau=0.0),
    "chain_f32": lambda: W.make_config(1, scale="small", device="cuda"),
    "medusa_232": lambda: _medusa(),
    "medusa_232_greedy": lambda: _medusa(tau=0.0),
    "medusa_f32_hot": lambda: _medusa(V=1999, dtype="f32", tau=1.6),
    "specinfer_321": lambda: _specinfer(),
    "specinfer_bf16_ragged": lambda: _specinfer(V=517, dtype="bf16", tau=1.0),
    "probs_f32": lambda: W.chain_workload(B=5, gamma=4, V=2003, dtype="f32", H_q=4, H_kv=4, d=64,
                                          prefix=40, tau=1.0, target_std=2.0, noise_std=1.0,
                                          device="cuda", draft_kind=W.DRAFT_PROBS),
    "probs_bf16": lambda: W.chain_workload(B=5, gamma=4, V=2003, dtype="bf16", H_q=4, H_kv=4,
                                           d=128, prefix=40, tau=1.0, target_std=2.0,
                                           noise_std=1.0, device="cuda",
                                           draft_kind=W.DRAFT_PROBS),
    "single_token_tiny_vocab": lambda: W.chain_workload(B=3, gamma=0, V=13, dtype="bf16", H_q=8,
                                                        H_kv=2, d=128, prefix=17, tau=1.0,
                                                        target_std=3.0, noise_std=1.0,
                                                        device="cuda", T_max=4),
    "many_requests": lambda: W.chain_workload(B=40, gamma=5, V=1001, dtype="bf16", H_q=4, H_kv=4,
                                              d=128, prefix=20, tau=1.0, target_std=2.0,
                                              noise_std=1.0, device="cuda"),
    # more clusters than the GPU holds at once: several waves
    "several_waves": lambda: W.chain_workload(B=200, gamma=3, V=517, dtype="bf16", H_q=4,
                                              H_kv=4, d=128, prefix=20, tau=1.0, target_std=2.0,
                                              noise_std=1.0, device="cuda"),
    # a 13-token vocabulary leaves most CTAs of a cluster without a slice
    "tiny_vocab_chain": lambda: W.chain_workload(B=4, gamma=4, V=13, dtype="bf16", H_q=4, H_kv=4,
                                                 d=128, prefix=17, tau=1.0, target_std=1.0,
                                                 noise_std=2.0, device="cuda"),
    "tiny_vocab_tree": lambda: _medusa(V=11, tau=0.8),
    # the largest trees the one-launch form takes: 32 nodes (a full warp of nodes)
    "chain_32_nodes": lambda: W.chain_workload(B=3, gamma=31, V=2003, dtype="bf16", H_q=4, H_kv=4,
                                               d=128, prefix=30, tau=1.0, target_std=1.0,
                                               noise_std=0.3, device="cuda"),
    "medusa_31_nodes": lambda: _medusa(V=1999, ks=(2, 2, 2, 2), B_=3),
}


def _verify(w, rule, path="cluster"):
    snap = PU.snapshot(w)
    step = VerifyStep(w, sibling_rule=rule, verify_path=PATHS[path])
    step.tree_build()
    step.verify()
    torch.cuda.synchronize()
    return step, snap


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_verify_paths_against_oracle(name, path):
    w = WORKLOADS[name]()
    step, snap = _verify(w, B.SPEC_SIBLING_RESIDUAL, path)
    PU.check_verify(w, step, PU.oracle_verify(w, snap))


@pytest.mark.parametrize("name", ["medusa_232", "specinfer_321"])
def test_independent_rule_paths(name, path):
    w = WORKLOADS[name]()
    step, snap = _verify(w, B.SPEC_SIBLING_INDEPENDENT, path)
    PU.check_verify(w, step, PU.oracle_verify(w, snap, B.SPEC_SIBLING_INDEPENDENT))


def test_the_forms_agree():
    # the three forms on the same inputs: every request's outputs are equal unless the oracle
    # itself puts one of its decisions within the fp32 band
    for name in ("medusa_232", "specinfer_321", "chain_bf16", "many_requests"):
        w = WORKLOADS[name]()
        outs = {}
        for p in ("cluster", "split", "walk"):
            step, snap = _verify(w, B.SPEC_SIBLING_RESIDUAL, p)
            outs[p] = {k: PU.np_(getattr(step, k)).copy()
                       for k in ("out_tokens", "out_len", "path", "n_acc", "rejections")}
        orc = PU.oracle_verify(w, snap)
        for other in ("split", "walk"):
            for r in range(w.B):
                same = all(np.array_equal(outs["cluster"][k][r], outs[other][k][r])
                           for k in outs[other])
                if not same:
                    events = orc["events"][r]
                    near = any((e[0] == "test" and abs(e[4] - e[3]) < PU.BAND) or
                               (e[0] == "sample" and e[3] < PU.BAND) for e in events)
                    assert near, (name, other, r)


def test_auto_takes_the_cluster_form_when_it_fits():
    # the one-launch form never touches the statistics workspace; the two-launch form fills it
    w = WORKLOADS["chain_bf16"]()
    for p, touched in (("cluster", False), ("split", True), ("walk", False)):
        step = VerifyStep(w, verify_path=PATHS[p])
        step.tree_build()
        step.ver_ws.fill_(0xA5)
        step.verify()
        torch.cuda.synchronize()
        assert bool((step.ver_ws != 0xA5).any()) == touched, p
    # a tree of more than 32 nodes takes the two-launch form below a vocabulary of 65536 and the
    # walk form from it (which never touches the statistics workspace)
    for V, touched in ((3001, True), (65536, False)):
        w = _medusa(V=V, ks=(3, 5, 7))   # 124 nodes
        step = VerifyStep(w)
        step.tree_build()
        step.ver_ws.fill_(0xA5)
        step.verify()
        torch.cuda.synchronize()
        assert bool((step.ver_ws != 0xA5).any()) == touched, V
        orc = PU.oracle_verify(w, PU.snapshot(w), B.SPEC_SIBLING_RESIDUAL)
        PU.check_verify(w, step, orc)


def _zero_q_workload(device="cuda"):
    """A Medusa (2, 3, 2) workload with draft probabilities in which some drafted tokens have
    draft probability exactly 0: in every request the root's second child (tested, after a
    rejection of the first, by the residual rule) and the first child of the root's first
    child (a plain ratio test)."""
    w = W.medusa_workload(B=6, ks=(2, 3, 2), V=3001, dtype="bf16", H_q=4, H_kv=4, d=128,
                          prefix=40, tau=1.0, device=device)
    V = w.V
    probs = torch.zeros(w.draft.shape, dtype=torch.float32, device=w.draft.device)
    probs[:, :V] = torch.softmax(w.draft[:, :V].float(), dim=-1)
    no, par = w.node_offset.cpu().numpy(), w.parent.cpu().numpy()
    tok, drow = w.tokens.cpu().numpy(), w.draft_row.cpu().numpy()
    for r in range(w.B):
        o, T = int(no[r]), int(no[r + 1] - no[r])
        kids = [[c for c in range(1, T) if par[o + c] == i] for i in range(T)]
        probs[int(drow[o]), int(tok[o + kids[0][1]])] = 0.0
        a = kids[0][0]
        probs[int(drow[o + a]), int(tok[o + kids[a][0]])] = 0.0
    w.draft = probs
    w.draft_kind = W.DRAFT_PROBS
    return w


def test_zero_draft_probability(path):
    # q(x) = 0 makes p / q = +inf: such a child is accepted whenever it is tested (its p is
    # positive), by the plain test and by the residual test alike
    w = _zero_q_workload()
    step, snap = _verify(w, B.SPEC_SIBLING_RESIDUAL, path)
    orc = PU.oracle_verify(w, snap)
    tested = [(r, e[2]) for r in range(w.B) for e in orc["events"][r]
              if e[0] == "test" and e[3] == np.inf]
    assert tested
    PU.check_verify(w, step, orc)
    path_of = PU.np_(step.path)
    for r, c in tested:
        assert c in path_of[r].tolist(), (r, c)


def _zero_mass_workload(device="cuda"):
    """A Medusa (2, 3, 2) workload with draft probabilities in which the root's draft row is
    q = 2 p_root (not normalised): the root's first child passes the ratio test iff
    u < p / q = 1/2, and after its rejection max(0, p - q) is 0 everywhere, so the final token
    is drawn from p.  The root's first child gets u = 0.75 (rejected) in even requests and 0.25
    (accepted) in odd ones."""
    w = W.medusa_workload(B=8, ks=(2, 3, 2), V=3001, dtype="bf16", H_q=4, H_kv=4, d=128,
                          prefix=40, tau=0.8, device=device)
    V = w.V
    probs = torch.zeros(w.draft.shape, dtype=torch.float32, device=w.draft.device)
    probs[:, :V] = torch.softmax(w.draft[:, :V].float(), dim=-1)
    no, par, drow = w.node_offset.cpu().numpy(), w.parent.cpu().numpy(), w.draft_row.cpu().numpy()
    for r in range(w.B):
        o = int(no[r])
        probs[int(drow[o]), :V] = 2.0 * torch.softmax(w.target[o, :V].float() / w.tau, dim=-1)
        first = next(c for c in range(1, int(no[r + 1]) - o) if par[o + c] == 0)
        w.uniforms[o + first, 0] = 0.75 if r % 2 == 0 else 0.25
    w.draft = probs
    w.draft_kind = W.DRAFT_PROBS
    return w


def test_zero_residual_mass_draws_from_p(path):
    w = _zero_mass_workload()
    step, snap = _verify(w, B.SPEC_SIBLING_RESIDUAL, path)
    orc = PU.oracle_verify(w, snap)
    for r in range(0, w.B, 2):   # the oracle stopped at the root after one rejection
        assert orc["path"][r] == [0] and orc["rejections"][r] == 1, r
    PU.check_verify(w, step, orc)


def test_data_errors_every_form(path):
    # a bad draft row and a bad token: flagged per request, outputs cleared, the other requests
    # verified as usual
    w = _medusa(B_=5)
    no = w.node_offset.cpu().numpy()
    internal = [i for i in range(no[1] - no[0]) if int(w.draft_row[no[0] + i]) >= 0]
    w.draft_row[no[0] + internal[1]] = w.R + 3
    w.tokens[no[1] + 4] = -2
    snap = PU.snapshot(w)
    step = VerifyStep(w, verify_path=PATHS[path])
    step.tree_build()
    step.verify()
    torch.cuda.synchronize()
    st = PU.np_(step.req_status)
    assert st[0] & B.REQ_BITS["BAD_DRAFT_ROW"]
    assert st[1] & B.REQ_BITS["BAD_TOKEN"]
    PU.check_verify(w, step, PU.oracle_verify(w, snap))


def _run_pair(make, fused):
    w = make()
    step = VerifyStep(w)
    step.tree_build()
    if fused:
        step.verify_compact()
    else:
        step.verify()
        step.compact()
    torch.cuda.synchronize()
    out = {k: PU.np_(getattr(step, k)).copy()
           for k in ("req_status", "out_tokens", "out_len", "path", "n_acc", "new_kv_len",
                     "slot_map", "blocks_in_use")}
    out["k"] = w.k_cache.float().cpu().numpy()
    out["v"] = w.v_cache.float().cpu().numpy()
    return out


def _bad_tree():
    w = _medusa(B_=5)
    no = w.node_offset.cpu().numpy()
    w.tokens[no[2] + 3] = w.V + 1
    P3 = int(w.prefix_len[3])
    w.block_table[3, P3 // w.bs] = w.k_cache.shape[1] + 9   # a tree slot's block out of range
    return w


FUSED = {
    "chain_2_layers": lambda: W.make_config(2, scale="small", device="cuda", num_layers=2),
    "medusa_2_layers": lambda: W.medusa_workload(B=4, ks=(2, 3, 2), V=3001, dtype="bf16", H_q=4,
                                                 H_kv=2, d=128, prefix=40, tau=1.0, device="cuda",
                                                 num_layers=2),
    "specinfer_f32": lambda: _specinfer(),
    "greedy_tree": lambda: _medusa(tau=0.0),
    "several_waves": WORKLOADS["several_waves"],
    "data_errors": _bad_tree,
    "tree_over_32_nodes": lambda: W.make_config(3, scale="small", device="cuda", num_layers=2),
}


@pytest.mark.parametrize("name", sorted(FUSED))
def test_verify_compact_equals_the_two_calls(name):
    # spec_verify_compact (compaction inside the one-launch verification, or launched after the
    # two-launch form) gives the same outputs and the same cache, byte for byte, as spec_verify
    # followed by spec_kv_compact
    a = _run_pair(FUSED[name], fused=False)
    b = _run_pair(FUSED[name], fused=True)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    if name == "data_errors":
        assert a["req_status"][2] & B.REQ_BITS["BAD_TOKEN"]
        assert a["req_status"][3] & B.REQ_BITS["BAD_BLOCK"]
    if name.startswith("medusa"):
        # accepted paths that are not the identity: slots were moved
        sm = a["slot_map"]
        assert ((sm[..., 0] >= 0) & (sm[..., 0] != sm[..., 1])).any()


def test_verify_compact_host_checks():
    w = WORKLOADS["chain_bf16"]()
    step = VerifyStep(w)
    other = torch.empty_like(step.path)
    bad = B.compact_params(w.k_cache, w.v_cache, w.block_table, w.prefix_len, other, step.n_acc,
                           step.req_status, step.new_kv_len, step.slot_map, step.blocks_in_use,
                           w.max_path)
    with pytest.raises(B.SpecError):
        B.spec_verify_compact(step.ver, bad, step.ver_ws)
