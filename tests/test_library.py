"""CPU-side checks of the C-ABI library: it builds for sm_103a, loads without a GPU, exports every
function include/spec_verify.h declares, and the Python structs match the C layouts."""
import ctypes
import os
import re
import subprocess

import pytest

from speculative_decoding_draft_tree_gb300 import binding as B
from speculative_decoding_draft_tree_gb300 import build

HEADER = os.path.join(build.INCLUDE, "spec_verify.h")


def declared_functions():
    with open(HEADER, encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return B.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"spec_tree_build", "spec_tree_attention", "spec_verify", "spec_kv_compact"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(B.EXPORTS) == set(names)


def test_status_strings(lib):
    for code, name in [(0, "SPEC_OK"), (1, "SPEC_ERR_INVALID_ARG"), (2, "SPEC_ERR_UNSUPPORTED"),
                       (3, "SPEC_ERR_CUDA")]:
        assert lib.spec_status_string(code).decode() == name


def test_struct_layouts_match_header(tmp_path):
    """Every field offset and every struct size of the Python binding equals what a C compiler
    makes of include/spec_verify.h."""
    structs = {"spec_attn_params": B.SpecAttnParams, "spec_verify_params": B.SpecVerifyParams,
               "spec_compact_params": B.SpecCompactParams, "spec_rope_params": B.SpecRopeParams,
               "spec_draft_pool": B.SpecDraftPool}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "spec_verify.h"',
             "int main(void) {"]
    want = []
    for cname, py in structs.items():
        lines.append(f'  printf("%zu\\n", sizeof({cname}));')
        want.append(ctypes.sizeof(py))
        for fname, _ in py._fields_:
            lines.append(f'  printf("%zu\\n", offsetof({cname}, {fname}));')
            want.append(getattr(py, fname).offset)
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    cc = subprocess.run(["gcc", "-I", build.INCLUDE, str(src), "-o", str(exe)],
                        capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    assert got == want


def test_constants_match_header(tmp_path):
    """Every status code, dtype, draft kind, sibling rule, verification form and request status
    bit the Python binding names has the value a C compiler gives it from the header."""
    consts = {"SPEC_OK": B.SPEC_OK, "SPEC_ERR_INVALID_ARG": B.SPEC_ERR_INVALID_ARG,
              "SPEC_ERR_UNSUPPORTED": B.SPEC_ERR_UNSUPPORTED, "SPEC_ERR_CUDA": B.SPEC_ERR_CUDA,
              "SPEC_F32": B.SPEC_F32, "SPEC_BF16": B.SPEC_BF16,
              "SPEC_DRAFT_LOGITS": B.SPEC_DRAFT_LOGITS, "SPEC_DRAFT_PROBS": B.SPEC_DRAFT_PROBS,
              "SPEC_SIBLING_RESIDUAL": B.SPEC_SIBLING_RESIDUAL,
              "SPEC_SIBLING_INDEPENDENT": B.SPEC_SIBLING_INDEPENDENT,
              "SPEC_SIBLING_MULTI_DRAFT": B.SPEC_SIBLING_MULTI_DRAFT,
              "SPEC_VERIFY_PATH_AUTO": B.SPEC_VERIFY_PATH_AUTO,
              "SPEC_VERIFY_PATH_SPLIT": B.SPEC_VERIFY_PATH_SPLIT,
              "SPEC_VERIFY_PATH_WALK": B.SPEC_VERIFY_PATH_WALK, "SPEC_MAX_TREE": B.SPEC_MAX_TREE}
    consts.update({f"SPEC_REQ_{k}": v for k, v in B.REQ_BITS.items()})
    lines = ["#include <stdio.h>", '#include "spec_verify.h"', "int main(void) {"]
    lines += [f'  printf("%d\\n", (int)({name}));' for name in consts]
    lines += ["  return 0;", "}"]
    src = tmp_path / "consts.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "consts"
    cc = subprocess.run(["gcc", "-I", build.INCLUDE, str(src), "-o", str(exe)],
                        capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    assert dict(zip(consts, got)) == consts


def test_host_validation_without_gpu(lib):
    # null parameter blocks are rejected before any CUDA call
    assert lib.spec_verify(None, None, 0, None) == B.SPEC_ERR_INVALID_ARG
    assert lib.spec_tree_attention(None, None, 0, None) == B.SPEC_ERR_INVALID_ARG
    assert lib.spec_kv_compact(None, None) == B.SPEC_ERR_INVALID_ARG
    assert lib.spec_tree_rope_kv_write(None, None) == B.SPEC_ERR_INVALID_ARG
    assert lib.spec_draft_init(None, None, None) == B.SPEC_ERR_INVALID_ARG
    assert lib.spec_echo_select_pack(None, 0, None, None, None, None, None, None, None, 0,
                                     None) == B.SPEC_ERR_INVALID_ARG
    assert lib.spec_echo_workspace_size(0, 0) == 0
    assert lib.spec_tree_build(None, None, None, 0, 0, 0, None, None, None, None, None,
                               None) == B.SPEC_ERR_INVALID_ARG
    assert lib.spec_verify_workspace_size(None) == 0


@pytest.mark.parametrize("change", [
    dict(B=0), dict(N=-1), dict(T_max=0), dict(T_max=257),   # outside [1, SPEC_MAX_TREE]
    dict(node_offset=None), dict(prefix_len=None), dict(req_status=None),
    dict(parent=None), dict(depth=None), dict(pos_id=None), dict(anc_mask=None),
    dict(is_internal=None),
])
def test_tree_build_host_validation(lib, change):
    fake = 0x100000   # never dereferenced: validation fails first
    a = dict(parent=fake, node_offset=fake, prefix_len=fake, B=2, N=8, T_max=6, depth=fake,
             pos_id=fake, anc_mask=fake, is_internal=fake, req_status=fake)
    a.update(change)
    assert lib.spec_tree_build(a["parent"], a["node_offset"], a["prefix_len"], a["B"], a["N"],
                               a["T_max"], a["depth"], a["pos_id"], a["anc_mask"],
                               a["is_internal"], a["req_status"], None) == B.SPEC_ERR_INVALID_ARG


def _rope(**kw):
    p = B.SpecRopeParams()
    p.dtype, p.B, p.N, p.H_q, p.H_kv, p.head_dim = B.SPEC_BF16, 2, 4, 4, 2, 128
    p.rotary_dim, p.interleaved, p.block_size, p.num_blocks, p.max_blocks_per_req = 128, 0, 16, 8, 4
    p.base = 10000.0
    fake = 0x100000   # 16-byte aligned, never dereferenced: validation fails first
    for f in ("q_in", "q_out", "k_new", "v_new", "k_cache", "v_cache", "block_table", "prefix_len",
              "node_offset", "pos_id", "req_status"):
        setattr(p, f, fake)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("change,code", [
    (dict(rotary_dim=127), B.SPEC_ERR_INVALID_ARG),          # odd
    (dict(rotary_dim=256), B.SPEC_ERR_INVALID_ARG),          # above head_dim
    (dict(rotary_dim=8), B.SPEC_ERR_UNSUPPORTED),            # half-split pair straddles vectors
    (dict(rotary_dim=12, interleaved=1), B.SPEC_ERR_UNSUPPORTED),
    (dict(base=0.0), B.SPEC_ERR_INVALID_ARG),
    (dict(base=float("inf")), B.SPEC_ERR_INVALID_ARG),
    (dict(head_dim=100), B.SPEC_ERR_INVALID_ARG),            # 200-byte rows: not 16-byte multiples
    (dict(q_out=0x100004), B.SPEC_ERR_INVALID_ARG),          # misaligned
    (dict(N=-1), B.SPEC_ERR_INVALID_ARG),
])
def test_rope_host_validation(lib, change, code):
    p = _rope(**change)
    assert lib.spec_tree_rope_kv_write(ctypes.byref(p), None) == code


def _attn(**kw):
    p = B.SpecAttnParams()
    p.dtype, p.B, p.N, p.T_max, p.H_q, p.H_kv, p.head_dim = B.SPEC_BF16, 2, 8, 6, 8, 2, 128
    p.block_size, p.num_blocks, p.max_blocks_per_req, p.scale = 16, 8, 4, 128 ** -0.5
    fake = 0x100000   # 16-byte aligned, never dereferenced: validation fails first
    for f in ("q", "k_cache", "v_cache", "block_table", "prefix_len", "node_offset", "anc_mask",
              "o", "req_status"):
        setattr(p, f, fake)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("change", [
    dict(dtype=7), dict(B=0), dict(N=-1), dict(T_max=0), dict(T_max=257),   # above SPEC_MAX_TREE
    dict(H_q=6, H_kv=4),                      # query heads not a multiple of the KV heads
    dict(head_dim=100),                       # 200-byte rows: not 16-byte multiples
    dict(dtype=B.SPEC_F32, head_dim=2),       # 8-byte rows
    dict(block_size=0), dict(num_blocks=0), dict(max_blocks_per_req=0),
    dict(q=0x100008), dict(k_cache=0x100004), dict(v_cache=0x100002), dict(o=0x100001),
    dict(q=None), dict(anc_mask=None), dict(block_table=None), dict(req_status=None),
])
def test_attention_host_validation(lib, change):
    p = _attn(**change)
    assert lib.spec_tree_attention(ctypes.byref(p), 0x100000, 1 << 30, None) == B.SPEC_ERR_INVALID_ARG
    assert lib.spec_attention_workspace_size(ctypes.byref(p)) == 0


def test_attention_with_no_nodes_is_a_no_op(lib):
    # N = 0: nothing to attend, the call succeeds before any CUDA call whatever the tensors
    p = _attn(N=0, q=None, k_cache=None, v_cache=None, o=None, anc_mask=None)
    assert lib.spec_tree_attention(ctypes.byref(p), None, 0, None) == B.SPEC_OK


def test_fused_rope_build_checks_its_request_arrays(lib):
    p = _rope()
    fake = 0x100000
    # the rope block's B / N must be the call's; a different node_offset buffer is refused
    assert lib.spec_tree_build_rope_kv_write(fake, fake, fake, 3, 4, 8, fake, fake, fake, fake,
                                             fake, ctypes.byref(p), None) == B.SPEC_ERR_INVALID_ARG
    p.node_offset = 0x200000
    assert lib.spec_tree_build_rope_kv_write(fake, fake, fake, 2, 4, 8, fake, fake, fake, fake,
                                             fake, ctypes.byref(p), None) == B.SPEC_ERR_INVALID_ARG


def test_draft_tree_host_validation(lib):
    fake = 0x100000
    pool = B.SpecDraftPool()
    pool.B, pool.cap = 4, 300   # above 256 candidates per request
    for f in ("parent", "token", "depth", "score", "row", "count"):
        setattr(pool, f, fake)
    assert lib.spec_draft_init(ctypes.byref(pool), fake, None) == B.SPEC_ERR_INVALID_ARG
    pool.cap = 100
    assert lib.spec_draft_expand_select(ctypes.byref(pool), 1, 17, fake, None,
                                        None) == B.SPEC_ERR_INVALID_ARG   # K above 16
    assert lib.spec_draft_topk_append(ctypes.byref(pool), 1, 5, fake, B.SPEC_BF16, fake, 1000,
                                      1000, 0.0, 0, None, None) == B.SPEC_ERR_INVALID_ARG  # tau
    assert lib.spec_draft_topk_append(ctypes.byref(pool), 1, 5, fake, B.SPEC_BF16, fake, 999,
                                      1000, 1.0, 0, None, None) == B.SPEC_ERR_INVALID_ARG  # ld < V
    assert lib.spec_echo_select_pack(ctypes.byref(pool), 64, fake, fake, fake, fake, fake, None,
                                     fake, 16, None) == B.SPEC_ERR_INVALID_ARG   # small workspace


def test_verify_path_field_is_validated(lib):
    # the form of the verification is chosen per call; values other than AUTO / SPLIT / WALK
    # are refused before any CUDA call
    v, _ = _fake_verify_and_compact()
    for bad in (-1, 3, 7):
        v.verify_path = bad
        assert lib.spec_verify(ctypes.byref(v), 0x100000, 1 << 30, None) == B.SPEC_ERR_INVALID_ARG


def _fake_verify_and_compact():
    fake = 0x100000   # 256-byte aligned, never dereferenced: validation fails first
    v = B.SpecVerifyParams()
    v.logits_dtype, v.draft_kind, v.sibling_rule = B.SPEC_BF16, B.SPEC_DRAFT_LOGITS, 0
    v.B, v.N, v.R, v.V, v.target_ld, v.draft_ld, v.T_max, v.max_path, v.tau = (
        2, 12, 10, 32000, 32000, 32000, 6, 6, 1.0)
    for f in ("target", "draft", "draft_row", "tokens", "parent", "node_offset", "depth",
              "is_internal", "uniforms", "req_status", "out_tokens", "out_len", "path", "n_acc",
              "rejections"):
        setattr(v, f, fake)
    c = B.SpecCompactParams()
    c.dtype, c.B, c.H_kv, c.head_dim, c.block_size = B.SPEC_BF16, 2, 4, 128, 16
    c.num_blocks, c.max_blocks_per_req, c.num_layers, c.max_path, c.layer_stride = 64, 32, 1, 6, 0
    for f in ("k_cache", "v_cache", "block_table", "prefix_len", "path", "n_acc", "req_status",
              "new_kv_len", "slot_map", "blocks_in_use"):
        setattr(c, f, fake)
    return v, c


@pytest.mark.parametrize("change", [
    dict(B=0), dict(N=-1), dict(R=-1), dict(V=0), dict(T_max=0), dict(T_max=257), dict(max_path=0),
    dict(tau=-0.5), dict(tau=float("nan")), dict(tau=float("inf")),
    dict(logits_dtype=5), dict(draft_kind=2), dict(sibling_rule=3),
    dict(target_ld=31999),                              # a row shorter than the vocabulary
    dict(target_ld=32001, draft_ld=32008),              # bf16 rows not 16-byte multiples
    dict(draft_ld=31992),
    dict(draft_kind=B.SPEC_DRAFT_PROBS, draft_ld=32002),   # fp32 rows of 128008 bytes
    dict(target=0x100008), dict(draft=0x100004), dict(draft=None),
    dict(tokens=None), dict(uniforms=None), dict(out_len=None), dict(n_acc=None),
])
def test_verify_host_validation(lib, change):
    # every field is checked before any CUDA call
    v, _ = _fake_verify_and_compact()
    for k, val in change.items():
        setattr(v, k, val)
    assert lib.spec_verify(ctypes.byref(v), 0x100000, 1 << 30, None) == B.SPEC_ERR_INVALID_ARG


def test_verify_workspace_checks(lib):
    # too small, not 256-byte aligned or missing: refused before any CUDA call
    v, _ = _fake_verify_and_compact()
    need = lib.spec_verify_workspace_size(ctypes.byref(v))
    assert need > 0
    assert lib.spec_verify(ctypes.byref(v), 0x100000, need - 1, None) == B.SPEC_ERR_INVALID_ARG
    assert lib.spec_verify(ctypes.byref(v), 0x100080, need, None) == B.SPEC_ERR_INVALID_ARG
    assert lib.spec_verify(ctypes.byref(v), None, need, None) == B.SPEC_ERR_INVALID_ARG


@pytest.mark.parametrize("change,code", [
    (dict(dtype=9), B.SPEC_ERR_INVALID_ARG), (dict(B=0), B.SPEC_ERR_INVALID_ARG),
    (dict(H_kv=0), B.SPEC_ERR_INVALID_ARG), (dict(block_size=0), B.SPEC_ERR_INVALID_ARG),
    (dict(num_layers=0), B.SPEC_ERR_INVALID_ARG), (dict(max_path=0), B.SPEC_ERR_INVALID_ARG),
    (dict(layer_stride=-8), B.SPEC_ERR_INVALID_ARG),
    (dict(layer_stride=4), B.SPEC_ERR_INVALID_ARG),     # 8 bytes between layers (bf16)
    (dict(head_dim=100), B.SPEC_ERR_INVALID_ARG),       # 200-byte rows
    (dict(k_cache=0x100008), B.SPEC_ERR_INVALID_ARG), (dict(v_cache=None), B.SPEC_ERR_INVALID_ARG),
    (dict(slot_map=None), B.SPEC_ERR_INVALID_ARG), (dict(blocks_in_use=None), B.SPEC_ERR_INVALID_ARG),
    (dict(num_layers=65536), B.SPEC_ERR_UNSUPPORTED),   # one grid row per layer
])
def test_kv_compact_host_validation(lib, change, code):
    _, c = _fake_verify_and_compact()
    for k, val in change.items():
        setattr(c, k, val)
    assert lib.spec_kv_compact(ctypes.byref(c), None) == code


@pytest.mark.parametrize("change", [dict(path=0x200000), dict(n_acc=0x200000),
                                    dict(req_status=0x200000), dict(B=3), dict(max_path=7),
                                    dict(head_dim=100)])
def test_verify_compact_host_validation(lib, change):
    # the compaction must read the verification's own results; mismatches are refused before
    # any CUDA call
    v, c = _fake_verify_and_compact()
    for k, val in change.items():
        setattr(c, k, val)
    ws, wsz = 0x100000, 1 << 30
    assert lib.spec_verify_compact(ctypes.byref(v), ctypes.byref(c), ws, wsz,
                                   None) == B.SPEC_ERR_INVALID_ARG
    assert lib.spec_verify_compact(ctypes.byref(v), None, ws, wsz, None) == B.SPEC_ERR_INVALID_ARG


C_CALLER = r"""
#include <stdio.h>
#include <string.h>
#include "spec_verify.h"

/* a plain C caller: status strings, and entry points that refuse their arguments before any
   CUDA call (so this runs without a GPU) */
int main(void) {
  int fails = 0;
  if (strcmp(spec_status_string(SPEC_OK), "SPEC_OK") != 0) ++fails;
  if (spec_verify(NULL, NULL, 0, NULL) != SPEC_ERR_INVALID_ARG) ++fails;
  if (spec_verify_compact(NULL, NULL, NULL, 0, NULL) != SPEC_ERR_INVALID_ARG) ++fails;
  {
    spec_verify_params v;
    memset(&v, 0, sizeof(v));
    if (v.verify_path != SPEC_VERIFY_PATH_AUTO) ++fails;   /* zero-initialised: the default */
    v.verify_path = 7;
    if (spec_verify(&v, NULL, 0, NULL) != SPEC_ERR_INVALID_ARG) ++fails;
  }
  if (spec_kv_compact(NULL, NULL) != SPEC_ERR_INVALID_ARG) ++fails;
  if (spec_tree_attention(NULL, NULL, 0, NULL) != SPEC_ERR_INVALID_ARG) ++fails;
  if (spec_verify_workspace_size(NULL) != 0) ++fails;
  printf("%d\n", fails);
  return fails;
}
"""


def test_plain_c_caller_links_and_runs(tmp_path, lib):
    # the boundary is a C ABI: a C program compiled against the header links the shared library
    # and calls it (validation paths only, no GPU needed)
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(build.LIB_PATH)
    cc = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", build.INCLUDE, str(src),
                         "-L", libdir, "-lspecverify", "-Wl,-rpath," + libdir, "-o", str(exe)],
                        capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0 and run.stdout.strip() == "0", (run.stdout, run.stderr)
