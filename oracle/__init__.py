"""CPU oracle for the draft-tree verification step -- TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 restatement of what the verification step computes, written from the pages'
definitions.  It shares no code with the CUDA library (no kernels, headers, helpers, tables or
constants) and never imports it.  Only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline / reference arm may import, call or execute anything in this package; the product path
(the C-ABI library and its Python binding) never does, and fails loudly when its CUDA extension
is missing.

Modules (each function cites the passage it follows):
  tree       -- flattening + ancestor mask + depth / position ids + internal-node flags
  attention  -- dense softmax attention of every tree token over prefix + its ancestors
  verify     -- temperature softmax, min(1, p/q) ratio test in tree order, residual resampling,
                bonus token, greedy (tau = 0) argmax matching
  compact    -- KV commit/rollback of the accepted path
  rope       -- rotary position embedding at the tree's position ids and the tree K/V written
                into its paged cache slots (the step before attention)
  lookahead  -- the lookahead-decoding mask (lookahead and verify branches in one forward)
  draft_tree -- building the draft tree: EAGLE-2 expansion of the most probable leaves, top-K
                of each expanded row, ECHO's batch-wide budget, packing for verification

Pins (tests/test_oracle_*.py, run with -m "not gpu") tie each function to something other than
itself: the page's 6-node mask table, the 123 / 45 node counts, E[L] = (1 - a^(g+1)) / (1 - a),
exact losslessness by black-box bisection over the uniforms, chi-square against p, library
scaled-dot-product attention for the T = 1 and chain special cases, the sequential-decoding
invariant for compaction, and RoFormer's complex form, the frequencies as numbers, brute force
over cache rows and chain = causal decoding for the RoPE step; a hand-derived worked example,
the page's token counts and its two mask rules for the lookahead mask; scipy's log_softmax, a
brute-force top-K, path products recomputed by multiplying probabilities, the page's node counts
and ECHO's optimality / ancestor closure for the draft-tree construction.
tests/test_oracle_mutations.py plants 73 plausible mistakes, one at a time, in fresh copies of
these modules, and each makes a named pin fail.  No oracle function is "parity unpinned".
"""
from . import tree, attention, verify, compact, rope, lookahead, draft_tree  # noqa: F401

# request status bits (the oracle's own numbering of the data errors it detects)
BAD_PARENT = 1
BAD_SIZE = 2
BAD_TOKEN = 4
BAD_DRAFT_ROW = 8
BAD_DEPTH = 16
BAD_BLOCK = 32
