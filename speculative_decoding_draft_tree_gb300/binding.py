"""Thin Python binding of the C-ABI in include/spec_verify.h (ctypes; argument marshalling only).

Every function here has the name of the C entry point it wraps, takes torch tensors that already
live on the GPU (device memory and streams are the only things torch provides), checks dtype /
device / contiguity, and calls the library on the current CUDA stream.  All computation happens
in the library's kernels; there is no CPU or PyTorch fallback: if libspecverify.so is missing or
fails to load, every call raises.
"""
import ctypes
import os

import torch

from . import build as _build

SPEC_OK, SPEC_ERR_INVALID_ARG, SPEC_ERR_UNSUPPORTED, SPEC_ERR_CUDA = 0, 1, 2, 3
SPEC_F32, SPEC_BF16 = 0, 1
SPEC_DRAFT_LOGITS, SPEC_DRAFT_PROBS = 0, 1
SPEC_SIBLING_RESIDUAL, SPEC_SIBLING_INDEPENDENT, SPEC_SIBLING_MULTI_DRAFT = 0, 1, 2
SPEC_VERIFY_PATH_AUTO, SPEC_VERIFY_PATH_SPLIT, SPEC_VERIFY_PATH_WALK = 0, 1, 2
SPEC_MAX_TREE = 256
REQ_BITS = dict(BAD_PARENT=1, BAD_SIZE=2, BAD_TOKEN=4, BAD_DRAFT_ROW=8, BAD_DEPTH=16,
                BAD_BLOCK=32, TIMEOUT=64)
EXPORTS = ["spec_tree_build", "spec_tree_rope_kv_write", "spec_tree_build_rope_kv_write", "spec_tree_attention", "spec_attention_workspace_size",
           "spec_verify", "spec_verify_workspace_size", "spec_verify_noalloc", "spec_kv_compact",
           "spec_status_string", "spec_last_cuda_error", "spec_draft_init",
           "spec_draft_expand_select", "spec_draft_topk_append", "spec_echo_workspace_size",
           "spec_echo_select_pack", "spec_debug_draft_copy_stall", "spec_verify_compact",
           "spec_kernel_launches"]

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64


class SpecAttnParams(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("B", _i32), ("N", _i32), ("T_max", _i32),
                ("H_q", _i32), ("H_kv", _i32), ("head_dim", _i32), ("block_size", _i32),
                ("num_blocks", _i32), ("max_blocks_per_req", _i32), ("scale", ctypes.c_float),
                ("q", _vp), ("k_cache", _vp), ("v_cache", _vp), ("block_table", _vp),
                ("prefix_len", _vp), ("node_offset", _vp), ("anc_mask", _vp), ("o", _vp),
                ("lse", _vp), ("req_status", _vp)]


class SpecVerifyParams(ctypes.Structure):
    _fields_ = [("logits_dtype", ctypes.c_int), ("draft_kind", ctypes.c_int),
                ("sibling_rule", ctypes.c_int), ("B", _i32), ("N", _i32), ("R", _i32),
                ("V", _i32), ("target_ld", _i64), ("draft_ld", _i64), ("T_max", _i32),
                ("max_path", _i32), ("tau", ctypes.c_float), ("target", _vp), ("draft", _vp),
                ("draft_row", _vp), ("tokens", _vp), ("parent", _vp), ("node_offset", _vp),
                ("depth", _vp), ("is_internal", _vp), ("uniforms", _vp), ("req_status", _vp),
                ("out_tokens", _vp), ("out_len", _vp), ("path", _vp), ("n_acc", _vp),
                ("rejections", _vp), ("verify_path", _i32)]


class SpecCompactParams(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("B", _i32), ("H_kv", _i32), ("head_dim", _i32),
                ("block_size", _i32), ("num_blocks", _i32), ("max_blocks_per_req", _i32),
                ("num_layers", _i32), ("max_path", _i32), ("layer_stride", _i64),
                ("k_cache", _vp), ("v_cache", _vp), ("block_table", _vp), ("prefix_len", _vp),
                ("path", _vp), ("n_acc", _vp), ("req_status", _vp), ("new_kv_len", _vp),
                ("slot_map", _vp), ("blocks_in_use", _vp)]


class SpecRopeParams(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("B", _i32), ("N", _i32), ("H_q", _i32), ("H_kv", _i32),
                ("head_dim", _i32), ("rotary_dim", _i32), ("interleaved", _i32),
                ("block_size", _i32), ("num_blocks", _i32), ("max_blocks_per_req", _i32),
                ("base", ctypes.c_double), ("q_in", _vp), ("q_out", _vp), ("k_new", _vp),
                ("v_new", _vp), ("k_cache", _vp), ("v_cache", _vp), ("block_table", _vp),
                ("prefix_len", _vp), ("node_offset", _vp), ("pos_id", _vp), ("req_status", _vp)]


class SpecDraftPool(ctypes.Structure):
    _fields_ = [("B", _i32), ("cap", _i32), ("parent", _vp), ("token", _vp), ("depth", _vp),
                ("score", _vp), ("row", _vp), ("count", _vp)]


_LIB = None


def library_path():
    return _build.LIB_PATH


def load_library(build_if_missing=False):
    """Load libspecverify.so (building it first when asked); raises if it cannot be loaded."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if build_if_missing and not _build.up_to_date():
        _build.build_library()
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    st = ctypes.c_int
    lib.spec_tree_build.restype = st
    lib.spec_tree_build.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.spec_tree_rope_kv_write.restype = st
    lib.spec_tree_build_rope_kv_write.restype = st
    lib.spec_tree_build_rope_kv_write.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp,
                                                  _vp, _vp, ctypes.POINTER(SpecRopeParams), _vp]
    lib.spec_tree_rope_kv_write.argtypes = [ctypes.POINTER(SpecRopeParams), _vp]
    lib.spec_tree_attention.restype = st
    lib.spec_tree_attention.argtypes = [ctypes.POINTER(SpecAttnParams), _vp, ctypes.c_size_t, _vp]
    lib.spec_attention_workspace_size.restype = ctypes.c_size_t
    lib.spec_attention_workspace_size.argtypes = [ctypes.POINTER(SpecAttnParams)]
    lib.spec_verify.restype = st
    lib.spec_verify.argtypes = [ctypes.POINTER(SpecVerifyParams), _vp, ctypes.c_size_t, _vp]
    lib.spec_verify_noalloc.restype = st
    lib.spec_verify_noalloc.argtypes = [ctypes.POINTER(SpecVerifyParams), _vp]
    lib.spec_verify_workspace_size.restype = ctypes.c_size_t
    lib.spec_verify_workspace_size.argtypes = [ctypes.POINTER(SpecVerifyParams)]
    lib.spec_kv_compact.restype = st
    lib.spec_kv_compact.argtypes = [ctypes.POINTER(SpecCompactParams), _vp]
    lib.spec_draft_init.restype = st
    lib.spec_draft_init.argtypes = [ctypes.POINTER(SpecDraftPool), _vp, _vp]
    lib.spec_draft_expand_select.restype = st
    lib.spec_draft_expand_select.argtypes = [ctypes.POINTER(SpecDraftPool), _i32, _i32, _vp, _vp,
                                             _vp]
    lib.spec_draft_topk_append.restype = st
    lib.spec_draft_topk_append.argtypes = [ctypes.POINTER(SpecDraftPool), _i32, _i32, _vp,
                                           ctypes.c_int, _vp, _i64, _i32, ctypes.c_float, _i32,
                                           _vp, _vp]
    lib.spec_debug_draft_copy_stall.restype = st
    lib.spec_debug_draft_copy_stall.argtypes = [_i32]
    lib.spec_verify_compact.restype = st
    lib.spec_verify_compact.argtypes = [ctypes.POINTER(SpecVerifyParams),
                                        ctypes.POINTER(SpecCompactParams), _vp, ctypes.c_size_t,
                                        _vp]
    lib.spec_echo_workspace_size.restype = ctypes.c_size_t
    lib.spec_echo_workspace_size.argtypes = [_i32, _i32]
    lib.spec_echo_select_pack.restype = st
    lib.spec_echo_select_pack.argtypes = [ctypes.POINTER(SpecDraftPool), _i32, _vp, _vp, _vp,
                                          _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.spec_kernel_launches.restype = ctypes.c_uint64
    lib.spec_kernel_launches.argtypes = []
    lib.spec_status_string.restype = ctypes.c_char_p
    lib.spec_status_string.argtypes = [ctypes.c_int]
    lib.spec_last_cuda_error.restype = ctypes.c_int
    lib.spec_last_cuda_error.argtypes = []
    _LIB = lib
    return lib


class SpecError(RuntimeError):
    pass


def _check(code, what):
    if code != SPEC_OK:
        lib = load_library()
        msg = lib.spec_status_string(code).decode()
        if code == SPEC_ERR_CUDA:
            msg += f" (cudaError {lib.spec_last_cuda_error()})"
        raise SpecError(f"{what}: {msg}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name, device=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise ValueError(f"unsupported dtype {t.dtype}")


# ----------------------------------------------------------------------------------------------
def spec_tree_build(parent, node_offset, prefix_len, T_max, depth, pos_id, anc_mask, is_internal,
                    req_status, stream=None):
    lib = load_library()
    i32 = torch.int32
    B = node_offset.numel() - 1
    N = parent.numel()
    for t, n in ((parent, "parent"), (node_offset, "node_offset"), (prefix_len, "prefix_len"),
                 (depth, "depth"), (pos_id, "pos_id"), (req_status, "req_status")):
        _need(t, i32, n)
    _need(anc_mask, torch.int32, "anc_mask")
    _need(is_internal, torch.uint8, "is_internal")
    code = lib.spec_tree_build(_ptr(parent), _ptr(node_offset), _ptr(prefix_len), B, N, T_max,
                               _ptr(depth), _ptr(pos_id), _ptr(anc_mask), _ptr(is_internal),
                               _ptr(req_status), _stream(stream))
    _check(code, "spec_tree_build")


def rope_params(q_in, q_out, k_new, v_new, k_cache, v_cache, block_table, prefix_len,
                node_offset, pos_id, req_status, base=10000.0, rotary_dim=None, interleaved=False):
    """k_cache / v_cache: one layer, [num_blocks, H_kv, block_size, head_dim]."""
    for t, n in ((q_in, "q_in"), (q_out, "q_out"), (k_new, "k_new"), (v_new, "v_new"),
                 (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, q_in.dtype, n)
    for t, n in ((block_table, "block_table"), (prefix_len, "prefix_len"),
                 (node_offset, "node_offset"), (pos_id, "pos_id"), (req_status, "req_status")):
        _need(t, torch.int32, n)
    p = SpecRopeParams()
    p.dtype = _dtype_code(q_in)
    p.B = node_offset.numel() - 1
    p.N, p.H_q, p.head_dim = q_in.shape
    p.H_kv = k_new.shape[1]
    if q_out.shape != q_in.shape or k_new.shape != (p.N, p.H_kv, p.head_dim) or v_new.shape != k_new.shape:
        raise ValueError("q_out must match q_in and v_new must match k_new [N, H_kv, head_dim]")
    p.rotary_dim = p.head_dim if rotary_dim is None else int(rotary_dim)
    p.interleaved = 1 if interleaved else 0
    p.num_blocks, _, p.block_size, _ = k_cache.shape
    p.max_blocks_per_req = block_table.shape[1]
    p.base = float(base)
    p.q_in, p.q_out, p.k_new, p.v_new = q_in.data_ptr(), q_out.data_ptr(), k_new.data_ptr(), v_new.data_ptr()
    p.k_cache, p.v_cache = k_cache.data_ptr(), v_cache.data_ptr()
    p.block_table, p.prefix_len = block_table.data_ptr(), prefix_len.data_ptr()
    p.node_offset, p.pos_id, p.req_status = node_offset.data_ptr(), pos_id.data_ptr(), req_status.data_ptr()
    return p


def spec_tree_build_rope_kv_write(parent, node_offset, prefix_len, T_max, depth, pos_id,
                                  anc_mask, is_internal, req_status, rope, stream=None):
    """spec_tree_build and spec_tree_rope_kv_write in one launch; `rope` from rope_params()
    over the same node_offset / prefix_len / pos_id / req_status."""
    lib = load_library()
    for t, n in ((parent, "parent"), (node_offset, "node_offset"), (prefix_len, "prefix_len"),
                 (depth, "depth"), (pos_id, "pos_id"), (req_status, "req_status"),
                 (anc_mask, "anc_mask")):
        _need(t, torch.int32, n)
    _need(is_internal, torch.uint8, "is_internal")
    code = lib.spec_tree_build_rope_kv_write(
        _ptr(parent), _ptr(node_offset), _ptr(prefix_len), node_offset.numel() - 1,
        parent.numel(), T_max, _ptr(depth), _ptr(pos_id), _ptr(anc_mask), _ptr(is_internal),
        _ptr(req_status), ctypes.byref(rope), _stream(stream))
    _check(code, "spec_tree_build_rope_kv_write")


def spec_tree_rope_kv_write(params, stream=None):
    code = load_library().spec_tree_rope_kv_write(ctypes.byref(params), _stream(stream))
    _check(code, "spec_tree_rope_kv_write")


def attention_params(q, k_cache, v_cache, block_table, prefix_len, node_offset, anc_mask, T_max,
                     o, lse, req_status, scale=0.0):
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (o, "o")):
        _need(t, None, n)
    for t, n in ((block_table, "block_table"), (prefix_len, "prefix_len"),
                 (node_offset, "node_offset"), (req_status, "req_status"),
                 (anc_mask, "anc_mask")):
        _need(t, torch.int32, n)
    if lse is not None:
        _need(lse, torch.float32, "lse")
    p = SpecAttnParams()
    p.dtype = _dtype_code(q)
    p.B = node_offset.numel() - 1
    p.N, p.H_q, p.head_dim = q.shape
    p.T_max = T_max
    p.num_blocks, p.H_kv, p.block_size = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    p.max_blocks_per_req = block_table.shape[1]
    p.scale = scale
    p.q, p.k_cache, p.v_cache = q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr()
    p.block_table, p.prefix_len = block_table.data_ptr(), prefix_len.data_ptr()
    p.node_offset, p.anc_mask = node_offset.data_ptr(), anc_mask.data_ptr()
    p.o = o.data_ptr()
    p.lse = None if lse is None else lse.data_ptr()
    p.req_status = req_status.data_ptr()
    return p


def spec_attention_workspace_size(params):
    return int(load_library().spec_attention_workspace_size(ctypes.byref(params)))


def spec_tree_attention(params, workspace, stream=None):
    lib = load_library()
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    code = lib.spec_tree_attention(ctypes.byref(params), _ptr(workspace), wsz, _stream(stream))
    _check(code, "spec_tree_attention")


def verify_params(target, draft, draft_kind, draft_row, tokens, parent, node_offset, depth,
                  is_internal, uniforms, tau, V, T_max, max_path, req_status, out_tokens,
                  out_len, path, n_acc, rejections=None, sibling_rule=SPEC_SIBLING_RESIDUAL,
                  verify_path=SPEC_VERIFY_PATH_AUTO):
    _need(target, None, "target")
    _need(draft, None, "draft")
    for t, n in ((draft_row, "draft_row"), (tokens, "tokens"), (parent, "parent"),
                 (node_offset, "node_offset"), (depth, "depth"), (req_status, "req_status"),
                 (out_tokens, "out_tokens"), (out_len, "out_len"), (path, "path"),
                 (n_acc, "n_acc")):
        _need(t, torch.int32, n)
    _need(is_internal, torch.uint8, "is_internal")
    _need(uniforms, torch.float32, "uniforms")
    p = SpecVerifyParams()
    p.logits_dtype = _dtype_code(target)
    p.draft_kind = draft_kind
    p.sibling_rule = sibling_rule
    p.B = node_offset.numel() - 1
    p.N = target.shape[0]
    p.R = draft.shape[0]
    p.V = V
    p.target_ld = target.shape[1]
    p.draft_ld = draft.shape[1]
    p.T_max, p.max_path, p.tau = T_max, max_path, float(tau)
    p.target, p.draft = target.data_ptr(), draft.data_ptr()
    p.draft_row, p.tokens, p.parent = draft_row.data_ptr(), tokens.data_ptr(), parent.data_ptr()
    p.node_offset, p.depth = node_offset.data_ptr(), depth.data_ptr()
    p.is_internal, p.uniforms = is_internal.data_ptr(), uniforms.data_ptr()
    p.req_status, p.out_tokens, p.out_len = req_status.data_ptr(), out_tokens.data_ptr(), out_len.data_ptr()
    p.path, p.n_acc = path.data_ptr(), n_acc.data_ptr()
    p.rejections = None if rejections is None else _need(rejections, torch.int32, "rejections").data_ptr()
    p.verify_path = int(verify_path)
    return p


def spec_verify_workspace_size(params):
    return int(load_library().spec_verify_workspace_size(ctypes.byref(params)))


def spec_verify(params, workspace, stream=None):
    lib = load_library()
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    code = lib.spec_verify(ctypes.byref(params), _ptr(workspace), wsz, _stream(stream))
    _check(code, "spec_verify")


def spec_verify_noalloc(params, stream=None):
    """spec_verify without a caller workspace (see include/spec_verify.h): for callers that may
    not allocate device memory.  Calls whose kernels overlap on the GPU share one scratch array
    and race."""
    code = load_library().spec_verify_noalloc(ctypes.byref(params), _stream(stream))
    _check(code, "spec_verify_noalloc")


def spec_verify_compact(vparams, cparams, workspace, stream=None):
    """spec_verify then spec_kv_compact in one call (one kernel when the verification takes its
    one-launch form); cparams must name vparams' path, n_acc and req_status."""
    lib = load_library()
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    code = lib.spec_verify_compact(ctypes.byref(vparams), ctypes.byref(cparams), _ptr(workspace),
                                   wsz, _stream(stream))
    _check(code, "spec_verify_compact")


def compact_params(k_cache, v_cache, block_table, prefix_len, path, n_acc, req_status,
                   new_kv_len, slot_map, blocks_in_use, max_path):
    """k_cache / v_cache: [L, num_blocks, H_kv, block_size, head_dim] (all layers)."""
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, None, n)
    for t, n in ((block_table, "block_table"), (prefix_len, "prefix_len"), (path, "path"),
                 (n_acc, "n_acc"), (req_status, "req_status"), (new_kv_len, "new_kv_len"),
                 (slot_map, "slot_map"), (blocks_in_use, "blocks_in_use")):
        _need(t, torch.int32, n)
    p = SpecCompactParams()
    p.dtype = _dtype_code(k_cache)
    L, nb, H_kv, bs, d = k_cache.shape
    p.B = block_table.shape[0]
    p.H_kv, p.head_dim, p.block_size, p.num_blocks = H_kv, d, bs, nb
    p.max_blocks_per_req = block_table.shape[1]
    p.num_layers, p.max_path = L, max_path
    p.layer_stride = nb * H_kv * bs * d
    p.k_cache, p.v_cache = k_cache.data_ptr(), v_cache.data_ptr()
    p.block_table, p.prefix_len = block_table.data_ptr(), prefix_len.data_ptr()
    p.path, p.n_acc, p.req_status = path.data_ptr(), n_acc.data_ptr(), req_status.data_ptr()
    p.new_kv_len, p.slot_map, p.blocks_in_use = new_kv_len.data_ptr(), slot_map.data_ptr(), blocks_in_use.data_ptr()
    return p


def spec_kv_compact(params, stream=None):
    code = load_library().spec_kv_compact(ctypes.byref(params), _stream(stream))
    _check(code, "spec_kv_compact")


# ----------------------------------------------------------------------------------------------
def draft_pool(parent, token, depth, score, row, count):
    """The candidate pool ([B, cap] int32 / fp32 arrays and count [B])."""
    for t, n in ((parent, "parent"), (token, "token"), (depth, "depth"), (row, "row"),
                 (count, "count")):
        _need(t, torch.int32, n)
    _need(score, torch.float32, "score")
    p = SpecDraftPool()
    p.B, p.cap = parent.shape
    p.parent, p.token, p.depth = parent.data_ptr(), token.data_ptr(), depth.data_ptr()
    p.score, p.row, p.count = score.data_ptr(), row.data_ptr(), count.data_ptr()
    return p


def spec_draft_init(pool, root_tokens, stream=None):
    _need(root_tokens, torch.int32, "root_tokens")
    _check(load_library().spec_draft_init(ctypes.byref(pool), _ptr(root_tokens), _stream(stream)),
           "spec_draft_init")


def spec_draft_expand_select(pool, level, K, expand, req_status=None, stream=None):
    _need(expand, torch.int32, "expand")
    code = load_library().spec_draft_expand_select(ctypes.byref(pool), level, K, _ptr(expand),
                                                   _ptr(req_status), _stream(stream))
    _check(code, "spec_draft_expand_select")


def spec_draft_topk_append(pool, level, K, expand, rows, V, tau, row_base, req_status=None,
                           stream=None):
    _need(expand, torch.int32, "expand")
    _need(rows, None, "rows")
    code = load_library().spec_draft_topk_append(ctypes.byref(pool), level, K, _ptr(expand),
                                                 _dtype_code(rows), _ptr(rows), rows.shape[1], V,
                                                 float(tau), row_base, _ptr(req_status),
                                                 _stream(stream))
    _check(code, "spec_draft_topk_append")


def spec_echo_workspace_size(B, cap):
    return int(load_library().spec_echo_workspace_size(B, cap))


def spec_echo_select_pack(pool, K_max, node_offset, parent, tokens, depth, draft_row, source,
                          workspace, stream=None):
    for t, n in ((node_offset, "node_offset"), (parent, "parent"), (tokens, "tokens"),
                 (depth, "depth"), (draft_row, "draft_row")):
        _need(t, torch.int32, n)
    wsz = workspace.numel() * workspace.element_size()
    code = load_library().spec_echo_select_pack(ctypes.byref(pool), K_max, _ptr(node_offset),
                                                _ptr(parent), _ptr(tokens), _ptr(depth),
                                                _ptr(draft_row), _ptr(source), _ptr(workspace),
                                                wsz, _stream(stream))
    _check(code, "spec_echo_select_pack")


def spec_debug_draft_copy_stall(chunk):
    """Testing only: make the next top-K launches lose one chunk's copy (-1: off)."""
    _check(load_library().spec_debug_draft_copy_stall(int(chunk)), "spec_debug_draft_copy_stall")


def spec_kernel_launches():
    """Kernels the library has enqueued in this process so far (a launch captured into a CUDA
    graph counts once, when captured; graph replays do not count)."""
    return int(load_library().spec_kernel_launches())
