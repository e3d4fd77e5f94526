"""Planted mistakes in the oracle, each caught by a committed pin.

Every case below copies one oracle module's source, makes one plausible mistake in it (a dropped
term, a wrong sign, index or scale, a transposed operand, a wrong tie rule), loads the copy as a
fresh module and runs the named pins of tests/test_oracle_*.py against it: at least one of them
must fail, by a failed comparison or by an error the mistake causes.  A control loads each
module unchanged the same way and every pin used here passes, so a failure comes from the
planted mistake, not from the loading.  Everything runs on the CPU; the library is never
involved.

Two changes are equivalent by construction and are not planted: the side of the inverse CDF's
search (it differs only on exact ties of u with a CDF edge, a set of measure zero) and an
in-place sequential copy in the compaction (equal to the gather because path[d] >= d).
"""
import importlib.util
import types

import numpy as np
import pytest

import test_oracle_attention as TA
import test_oracle_compact as TC
import test_oracle_draft_tree as TD
import test_oracle_lookahead as TL
import test_oracle_rope as TR
import test_oracle_tree as TT
import test_oracle_verify as TV
from oracle import verify as OV


def _load(modname, old=None, new=None):
    """A fresh copy of oracle.<modname>, with the one occurrence of `old` replaced by `new`."""
    spec = importlib.util.find_spec(f"oracle.{modname}")
    with open(spec.origin, encoding="utf-8") as f:
        src = f.read()
    if old is not None:
        assert src.count(old) == 1, f"{modname}: {old!r} occurs {src.count(old)} times"
        src = src.replace(old, new)
    m = types.ModuleType(f"oracle.{modname}")
    m.__package__ = "oracle"   # its relative imports resolve to the unchanged modules
    m.__file__ = spec.origin
    exec(compile(src, spec.origin, "exec"), m.__dict__)
    return m


# the test module and the name under which it holds each oracle module
HOLDER = {"verify": (TV, "OV"), "tree": (TT, "OT"), "attention": (TA, "OA"), "compact": (TC, "OC"),
          "lookahead": (TL, "OL"), "rope": (TR, "OR"), "draft_tree": (TD, "OD")}

# pins: (name, function, arguments)
LOSSLESS_SIBLINGS = ("exact losslessness, 3 siblings", TV.test_exact_losslessness,
                     ([-1, 0, 0, 0], 3, 1.0, OV.DRAFT_LOGITS))
LOSSLESS_PROBS = ("exact losslessness, draft probabilities", TV.test_exact_losslessness,
                  ([-1, 0, 0, 1], 3, 0.7, OV.DRAFT_PROBS))
LOSSLESS_CHAIN = ("exact losslessness, chain, tau 1.3", TV.test_exact_losslessness,
                  ([-1, 0, 1], 4, 1.3, OV.DRAFT_LOGITS))
LOSSLESS_MULTI = ("exact losslessness, multi-draft", TV.test_exact_losslessness_multi_draft,
                  ([-1, 0, 0, 0], 3, 1.0, OV.DRAFT_LOGITS))
LOSSLESS_MULTI2 = ("exact losslessness, multi-draft, two levels",
                   TV.test_exact_losslessness_multi_draft, ([-1, 0, 0, 1], 3, 0.7, OV.DRAFT_PROBS))
EXPECTED_L = ("E[L] closed form", TV.test_expected_emitted_length, (1, 0.2))
GREEDY_LIMIT = ("greedy is the tau -> 0+ limit", TV.test_greedy_is_the_low_temperature_limit, ())
GREEDY_TIES = ("greedy ties to the lowest id", TV.test_greedy_ties_go_to_lowest_token, ())
DATA_ERRORS = ("data errors flagged", TV.test_data_errors_flagged, ())
PAGE_MASK = ("the page's mask table", TT.test_page_mask_table_reproduced_exactly, ())
POS_IDS = ("position ids", TT.test_position_ids_are_prefix_plus_depth, ())
CHAIN_MASK = ("chain mask", TT.test_chain_mask_is_lower_triangular, ())
NODE_COUNTS = ("printed node counts", TT.test_printed_node_counts, ("medusa",))
DECODE = ("decode attention", TA.test_single_token_is_decode_attention, ())
KV_ONE = ("KV length one", TA.test_kv_length_one, ())
EXPLICIT_SCALE = ("explicit scale", TA.test_explicit_scale, ())
TREE_PATH = ("tree node = sequence over its path", TA.test_tree_node_equals_sequence_over_its_path, ())
CHAIN_CAUSAL = ("chain = causal attention", TA.test_chain_is_causal_attention, ())
SEQUENTIAL = ("compaction = sequential decoding", TC.test_compaction_equals_sequential_decoding, ())
ROLLBACK = ("rejected request rolls back", TC.test_rejected_request_rolls_back_everything, ())
LA_WORKED = ("worked lookahead example", TL.test_worked_example, ())
LA_RULES = ("lookahead rules", TL.test_rules, (5, 4, 5))
LA_ANCESTOR = ("lookahead ancestor mask", TL.test_is_an_ancestor_mask, (5, 4, 5))
LA_JACOBI = ("N = 2 is Jacobi decoding", TL.test_n2_is_jacobi_decoding, ())
ROPE_COMPLEX = ("RoFormer complex form", TR.test_complex_form, ())
ROPE_FREQ = ("frequencies as numbers", TR.test_frequencies_as_numbers, ())
ROPE_HALF = ("half-split = permuted interleaved", TR.test_half_split_is_permuted_interleaved, ())
ROPE_TAIL = ("partial rotary", TR.test_partial_rotary_leaves_tail, ())
ROPE_SLOTS = ("slot write brute force", TR.test_slot_write_brute_force, ())
ROPE_CHAIN = ("chain = causal decoding", TR.test_chain_equals_causal_decoding, ())
DT_TOPK = ("log_softmax and top-K", TD.test_log_softmax_and_topk, ())
DT_COUNTS = ("the page's counts", TD.test_counts_of_the_page, ())
DT_PATHS = ("most probable paths", TD.test_expanded_leaves_are_the_most_probable_paths, ())
DT_ECHO = ("ECHO budget", TD.test_echo_budget, (40,))
DT_ECHO_SMALL = ("ECHO budget, small", TD.test_echo_budget, (8,))
DT_CONFIDENT = ("confident requests", TD.test_confident_requests_get_the_budget, ())
DT_PACKED = ("packed layout", TD.test_packed_layout_is_a_tree, ())
GREEDY_TREE = ("greedy walk on a hand-made tree", TV.test_greedy_walk_on_a_hand_made_tree, ())
ZERO_Q = ("zero draft probability", TV.test_a_draft_token_with_zero_draft_probability, ())
CDF_GAP = ("inverse CDF and its edge distance", TV.test_inverse_cdf_and_its_distance_to_the_edges,
           ())
RATIOS = ("recorded ratios", TV.test_recorded_ratios_are_p_over_q, ())
ZERO_MASS = ("zero residual mass draws from p", TV.test_zero_residual_mass_draws_from_p,
             (OV.SIBLING_RESIDUAL,))
ZERO_MASS_MULTI = ("zero residual mass draws from p, multi-draft",
                   TV.test_zero_residual_mass_draws_from_p, (OV.SIBLING_MULTI_DRAFT,))
COMPACT_BAD = ("bad block rolls back", TC.test_bad_block_flagged, ())
DT_SCORES = ("scores at tau 0.5", TD.test_scores_are_path_log_probabilities, (0.5,))
DT_TIES = ("ECHO ties", TD.test_echo_ties_go_to_the_lower_request_then_the_lower_candidate, ())
INDEP_CHAIN = ("independent rule lossless on chains", TV.test_independent_rule_is_lossless_on_chains,
               (OV.DRAFT_LOGITS,))
ATTN_BAD_BLOCK = ("bad block flagged", TA.test_bad_block_flagged, ())
ROPE_SKIPS = ("skipped nodes and requests", TR.test_bad_block_and_bad_request_are_skipped, ())
TREE_INVALID = ("invalid trees flagged", TT.test_invalid_trees_flagged, ())

MUTATIONS = [
    # --- verification (ratio test, residual, draws) ---
    ("residual scale: C grows by 1 instead of N_k", "verify",
     "C = C + Nk", "C = C + 1.0", [LOSSLESS_SIBLINGS]),
    ("residual from the first rejection only", "verify",
     "Rk = p if C == 0.0 else np.maximum(0.0, p - C * q)", "Rk = p",
     [LOSSLESS_SIBLINGS]),
    ("ratio test against q instead of N_k q", "verify",
     "num, den = Rk[tok], Nk * q[tok]", "num, den = Rk[tok], q[tok]", [LOSSLESS_SIBLINGS]),
    ("final draw from p - q after several rejections", "verify",
     "(C if sibling_rule == SIBLING_RESIDUAL else 1.0) * q", "1.0 * q", [LOSSLESS_SIBLINGS]),
    ("off-by-one inverse CDF", "verify",
     "x = min(x, len(c) - 1)", "x = min(x + 1, len(c) - 1)", [LOSSLESS_CHAIN]),
    ("draft q without the temperature", "verify",
     "softmax_at(row, tau) if draft_kind", "softmax_at(row, 1.0) if draft_kind", [LOSSLESS_CHAIN]),
    ("bonus token drawn uniformly", "verify",
     "final, gap = inverse_cdf(p, u_samp)", "final, gap = inverse_cdf(np.ones_like(p), u_samp)",
     [LOSSLESS_CHAIN]),
    ("bonus token drawn from the parent's p", "verify",
     "p = softmax_at(target[o + node, :V], tau)\n            u_samp",
     "p = softmax_at(target[o + (node if kids_of[node] else path[-2]), :V], tau)\n            u_samp",
     [LOSSLESS_CHAIN]),
    ("acceptance test reversed (u > a)", "verify",
     "                if u < a:\n                    accepted = c\n                    break\n"
     "                rejections += 1\n                if sibling_rule == SIBLING_RESIDUAL:",
     "                if u > a:\n                    accepted = c\n                    break\n"
     "                rejections += 1\n                if sibling_rule == SIBLING_RESIDUAL:",
     [LOSSLESS_PROBS]),
    ("emitted length without the final token", "verify",
     'res["out_len"][r] = len(path)', 'res["out_len"][r] = len(path) - 1', [EXPECTED_L]),
    ("inverted greedy match", "verify",
     "if tokens[o + c] == best:", "if tokens[o + c] != best:", [GREEDY_LIMIT]),
    ("greedy ties to the highest id", "verify",
     "best = int(np.argmax(np.asarray(target[o + node, :V], dtype=np.float64)))",
     "best = int(V - 1 - np.argmax(np.asarray(target[o + node, :V], dtype=np.float64)[::-1]))",
     [GREEDY_TIES]),
    ("greedy rejections counted twice", "verify",
     "                    rejections += 1\n                if nxt is None:",
     "                    rejections += 2\n                if nxt is None:", [GREEDY_TREE]),
    ("q(x) = 0 read as a failed test", "verify",
     "num, den = p[tok], q[tok]\n                a = num / den if den > 0 else (np.inf if num > 0 else 0.0)",
     "num, den = p[tok], q[tok]\n                a = num / den if den > 0 else 0.0", [ZERO_Q]),
    ("greedy checks draft rows it never reads", "verify",
     "elif tau > 0 and any(kids_of[i] and", "elif any(kids_of[i] and", [DATA_ERRORS]),
    ("multi-draft checks the parents' rows", "verify",
     "if tau > 0 and any(not (0 <= draft_row[o + c] < R) for c in range(1, T)):",
     "if tau > 0 and any(kids_of[i] and not (0 <= draft_row[o + i] < R) for i in range(T)):",
     [DATA_ERRORS]),
    ("zero residual mass: final draw from the (empty) residual", "verify",
     "                    if Nk <= 0.0:\n                        w_final = p\n",
     "                    if Nk <= 0.0:\n                        w_final = np.maximum(0.0, p - C * q)\n",
     [ZERO_MASS]),
    ("multi-draft zero residual mass: final draw from the residual", "verify",
     "                    if mass <= 0.0:\n                        w_final = p\n",
     "                    if mass <= 0.0:\n                        w_final = resid\n", [ZERO_MASS_MULTI]),
    ("a draw's edge distance not normalised", "verify",
     "lo = c[x - 1] / total if x > 0 else 0.0", "lo = c[x - 1] if x > 0 else 0.0", [CDF_GAP]),
    ("every draw recorded far from an edge", "verify",
     "return x, min(u - lo, hi - u)", "return x, 1.0", [CDF_GAP]),
    ("recorded ratio clipped at 1", "verify",
     '                u = float(uniforms[o + c, 0])\n                events.append(("test", node, c, a, u))',
     '                u = float(uniforms[o + c, 0])\n                events.append(("test", node, c, min(a, 1.0), u))',
     [RATIOS]),
    ("token range check off by one", "verify",
     "not (0 <= tokens[o + c] < V)", "not (0 <= tokens[o + c] <= V)", [DATA_ERRORS]),
    ("independent rule resamples from p", "verify",
     "(C if sibling_rule == SIBLING_RESIDUAL else 1.0) * q",
     "(C if sibling_rule == SIBLING_RESIDUAL else 0.0) * q", [INDEP_CHAIN]),
    ("multi-draft: later siblings tested against p", "verify",
     "num, den = target_now[tok], qc[tok]", "num, den = p[tok], qc[tok]", [LOSSLESS_MULTI]),
    ("multi-draft: residual not renormalised", "verify",
     "target_now = resid / mass", "target_now = resid", [LOSSLESS_MULTI]),
    ("multi-draft: the parent's q instead of the child's", "verify",
     "qc = q_of(draft_row[o + c])", "qc = q_of(draft_row[o + node])", [LOSSLESS_MULTI2]),
    # --- tree build ---
    ("mask without the self bit", "tree", "for j in chain:", "for j in chain[1:]:", [PAGE_MASK]),
    ("mask with only the parent", "tree", "for j in chain:", "for j in chain[:2]:", [PAGE_MASK]),
    ("depth counted from 1", "tree",
     "depth[o + i] = len(chain) - 1", "depth[o + i] = len(chain)", [PAGE_MASK]),
    ("position id without the prefix", "tree",
     "pos_id[o + i] = int(prefix_len[r]) + depth[o + i]", "pos_id[o + i] = depth[o + i]",
     [POS_IDS]),
    ("children marked internal instead of parents", "tree",
     "is_internal[o + par[i]] = True", "is_internal[o + i] = True", [NODE_COUNTS]),
    ("mask transposed", "tree", "M[i, j] = True", "M[j, i] = True", [CHAIN_MASK]),
    ("the root's first child does not make it internal", "tree",
     "for i in range(1, T):\n            is_internal", "for i in range(2, T):\n            is_internal",
     [CHAIN_MASK]),
    ("size bound one too loose", "tree",
     "if T < 1 or T > T_max:", "if T < 1 or T > T_max + 1:", [TREE_INVALID]),
    # --- tree attention ---
    ("scale 1/d instead of 1/sqrt(d)", "attention",
     "scale = 1.0 / np.sqrt(d) if scale is None", "scale = 1.0 / d if scale is None", [DECODE]),
    ("lse without the maximum", "attention",
     "lse_out[n, h] = m + np.log(z)", "lse_out[n, h] = np.log(z)", [KV_ONE]),
    ("query head h reads KV head h mod H_kv", "attention",
     "K = _gather(kc, table[r], slots, h // G, bs)", "K = _gather(kc, table[r], slots, h % H_kv, bs)",
     [TREE_PATH]),
    ("a node does not see itself", "attention",
     "sorted(P + a for a in ancestors_or_self(par, i))",
     "sorted(P + a for a in ancestors_or_self(par, i)[1:])", [CHAIN_CAUSAL]),
    ("a caller's scale ignored", "attention",
     "scale = 1.0 / np.sqrt(d) if scale is None else scale", "scale = 1.0 / np.sqrt(d)",
     [EXPLICIT_SCALE]),
    ("lse in base 2", "attention",
     "lse_out[n, h] = m + np.log(z)", "lse_out[n, h] = m + np.log2(z)", [DECODE]),
    ("bad-block range rounded down", "attention",
     "nblk = -(-(P + T) // bs)", "nblk = (P + T) // bs", [ATTN_BAD_BLOCK]),
    ("K and V swapped", "attention",
     "o_out[n, h] = (w @ Vv) / z", "o_out[n, h] = (w @ K) / z", [DECODE]),
    # --- KV compaction ---
    ("source and destination transposed", "compact",
     "src, dst = P + pr[dd], P + dd", "src, dst = P + dd, P + pr[dd]", [SEQUENTIAL]),
    ("committed length without the last accepted slot", "compact",
     "new_len[r] = P + na + 1", "new_len[r] = P + na", [SEQUENTIAL]),
    ("a bad block's request releases its prefix blocks", "compact",
     "            status[r] |= BAD_BLOCK\n            blocks_in_use[r] = -(-P // bs)",
     "            status[r] |= BAD_BLOCK\n            blocks_in_use[r] = 0", [COMPACT_BAD]),
    ("a request with a data error keeps its accepted path", "compact",
     "if status[r] or na < 0:", "if na < 0:", [ROLLBACK]),
    # --- lookahead mask ---
    ("verify candidates see each other", "lookahead",
     "return ga == gb and kb < ka", "return kb < ka", [LA_WORKED]),
    ("rule 2 dropped", "lookahead", "if a[0] != b[0]:", "if False:", [LA_RULES]),
    ("step-0 token at position 1 not seen", "lookahead",
     "if lb == 0 and 1 <= pb < start:", "if lb == 0 and 2 <= pb < start:", [LA_RULES]),
    ("diagonal read as a column", "lookahead",
     "return lb < la and pb - lb == start", "return lb < la and pb == pa", [LA_ANCESTOR]),
    ("step 0 starts at position 0", "lookahead",
     'nodes += [("look", 0, p) for p in range(1, W)]',
     'nodes += [("look", 0, p) for p in range(0, W - 1)]', [LA_JACOBI]),
    # --- RoPE ---
    ("rotation clockwise", "rope",
     "c, s = np.cos(ang), np.sin(ang)", "c, s = np.cos(ang), -np.sin(ang)", [ROPE_FREQ]),
    ("frequency exponent without the 2", "rope",
     "theta = base ** (-2.0 * j / rotary_dim)", "theta = base ** (-1.0 * j / rotary_dim)",
     [ROPE_FREQ]),
    ("half-split pairs read as interleaved", "rope",
     "return [(j, j + half) for j in range(half)]",
     "return [(2 * j, 2 * j + 1) for j in range(half)]", [ROPE_HALF]),
    ("rotary_dim ignored (whole head rotated)", "rope",
     "rotary_dim = d if rotary_dim is None else int(rotary_dim)", "rotary_dim = d", [ROPE_TAIL]),
    ("slot off by one", "rope", "slot = P + i", "slot = P + i + 1", [ROPE_SLOTS]),
    ("negative position ids rotated", "rope",
     "            if m < 0:\n                continue\n", "", [ROPE_SKIPS]),
    ("k written unrotated", "rope",
     "kc[blk, :, row, :] = rope(k_new[n], m, base, rotary_dim, interleaved)",
     "kc[blk, :, row, :] = k_new[n]", [ROPE_CHAIN]),
    # --- draft tree construction ---
    ("log_softmax without the temperature", "draft_tree",
     "y = np.asarray(row, dtype=np.float64) / tau", "y = np.asarray(row, dtype=np.float64)",
     [DT_TOPK]),
    ("top-K ties to the higher id", "draft_tree",
     "key=lambda x: (-lq[x], x)", "key=lambda x: (-lq[x], -x)", [DT_TOPK]),
    ("top-K one short when K reaches the vocabulary", "draft_tree",
     "k = min(k, n)", "k = min(k, n - 1)", [DT_TOPK]),
    ("path score without the parent's score", "draft_tree",
     'score=cs[i]["score"] + float(lp)', "score=float(lp)", [DT_PATHS]),
    ("the K worst leaves expanded", "draft_tree",
     'best = sorted(front, key=lambda i: (-cs[i]["score"], i))[:K]',
     'best = sorted(front, key=lambda i: (cs[i]["score"], i))[:K]', [DT_PATHS]),
    ("one leaf too many expanded", "draft_tree",
     'best = sorted(front, key=lambda i: (-cs[i]["score"], i))[:K]',
     'best = sorted(front, key=lambda i: (-cs[i]["score"], i))[:K + 1]', [DT_COUNTS]),
    ("ECHO budget not net of the roots", "draft_tree",
     "nonroot[:max(0, K_max - pool.B)]", "nonroot[:max(0, K_max)]", [DT_ECHO]),
    ("ECHO drops the roots", "draft_tree",
     "keep = set((r, 0) for r in range(pool.B)) | set(", "keep = set() | set(", [DT_ECHO_SMALL]),
    ("ECHO keeps the least probable", "draft_tree",
     'nonroot.sort(key=lambda ri: (-pool.cands[ri[0]][ri[1]]["score"], ri[0], ri[1]))',
     'nonroot.sort(key=lambda ri: (pool.cands[ri[0]][ri[1]]["score"], ri[0], ri[1]))',
     [DT_CONFIDENT]),
    ("top-K at tau 1 whatever the temperature", "draft_tree",
     "tops = [[topk(rows[r][j], K, tau)", "tops = [[topk(rows[r][j], K)", [DT_SCORES]),
    ("an expanded candidate's children in reverse order", "draft_tree",
     "for t, lp in zip(toks, lps):", "for t, lp in list(zip(toks, lps))[::-1]:", [DT_SCORES]),
    ("root score 1", "draft_tree",
     'depth=0, score=0.0, row=-1', 'depth=0, score=1.0, row=-1', [DT_SCORES]),
    ("ECHO ties to the higher request", "draft_tree",
     '["score"], ri[0], ri[1]))', '["score"], -ri[0], ri[1]))', [DT_TIES]),
    ("ECHO ties to the higher candidate", "draft_tree",
     '["score"], ri[0], ri[1]))', '["score"], ri[0], -ri[1]))', [DT_TIES]),
    ("draft row kept on nodes with no kept child", "draft_tree",
     'draft_row.append(c["row"] if old in has_kept_child else -1)', 'draft_row.append(c["row"])',
     [DT_PACKED]),
]


def _run_pins(modname, module, pins, monkeypatch):
    """The names of the pins that fail with `module` standing in for oracle.<modname>."""
    holder, attr = HOLDER[modname]
    failed = []
    for name, fn, args in pins:
        # a planted mistake may divide by a zero mass: its warnings are expected
        with monkeypatch.context() as mp, np.errstate(all="ignore"):
            mp.setattr(holder, attr, module)
            try:
                fn(*args)
            except Exception:   # a failed comparison, or the mistake breaking the computation
                failed.append(name)
    return failed


@pytest.mark.parametrize("modname", sorted(HOLDER))
def test_unchanged_copies_pass_every_pin(modname, monkeypatch):
    pins = {p[0]: p for m in MUTATIONS if m[1] == modname for p in m[4]}
    assert pins
    assert _run_pins(modname, _load(modname), list(pins.values()), monkeypatch) == []


@pytest.mark.parametrize("what,modname,old,new,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(what, modname, old, new, pins, monkeypatch):
    assert _run_pins(modname, _load(modname, old, new), pins, monkeypatch), what
