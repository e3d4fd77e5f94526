"""One verification round on the GPU through the C-ABI: tree build -> tree attention (one layer)
-> verify -> KV compaction.

`VerifyStep` owns every output and workspace buffer for a fixed workload shape (allocated once
with torch, never inside the timed calls) and runs the four library calls on the current stream.
`run_from_host` is the end-to-end form: the step's inputs arrive in pinned host memory, are
copied to the device, the round runs, and the accepted tokens come back to the host.  For a
stream of rounds, `twin()` gives a second step over its own copies of the per-round inputs (same
KV cache), so that one step's `upload` on a copy stream overlaps the other's `run`.
"""
import dataclasses
from dataclasses import dataclass
from typing import Dict, Optional

import torch

from . import binding as B
from .workloads import Workload


def _ws(nbytes: int, device) -> torch.Tensor:
    # torch allocations are 256-byte aligned (caching allocator) -- the library checks it
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _packed(tensors: Dict[str, torch.Tensor], device, pin: bool = False):
    """One contiguous byte buffer holding tensors shaped like `tensors` at 256-byte aligned
    offsets, and the views into it (one copy moves them all)."""
    offs, off = {}, 0
    for k, t in tensors.items():
        off = (off + 255) // 256 * 256
        offs[k] = off
        off += t.numel() * t.element_size()
    buf = torch.empty(max(off, 1), dtype=torch.uint8, device=device)
    if pin:
        buf = buf.pin_memory()
    views = {k: buf[offs[k]:offs[k] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
             for k, t in tensors.items()}
    return buf, views


class VerifyStep:
    """One verification round's outputs, workspaces and C-ABI parameter blocks over a workload's
    device tensors.  verify_path is SPEC_VERIFY_PATH_AUTO (the form is chosen per call from the
    tree sizes and the vocabulary), _SPLIT (row statistics kernel, then the walk) or _WALK (the
    walk forms the statistics of the nodes it visits)."""

    def __init__(self, w: Workload, sibling_rule: int = B.SPEC_SIBLING_RESIDUAL,
                 with_lse: bool = True, verify_path: int = B.SPEC_VERIFY_PATH_AUTO):
        self.w = w
        self.sibling_rule = sibling_rule
        self.verify_path = verify_path
        dev = w.target.device
        if dev.type != "cuda":
            raise ValueError("VerifyStep needs the workload on a CUDA device")
        i32 = dict(dtype=torch.int32, device=dev)
        Bn, N, W = w.B, w.N, (w.T_max + 31) // 32
        self.req_status = torch.zeros(Bn, **i32)
        self.depth = torch.empty(N, **i32)
        self.pos_id = torch.empty(N, **i32)
        self.anc_mask = torch.empty((N, W), **i32)
        self.is_internal = torch.empty(N, dtype=torch.uint8, device=dev)
        self.o = torch.empty_like(w.q)
        self.lse = torch.empty((N, w.H_q), dtype=torch.float32, device=dev) if with_lse else None
        # the results a round sends back to the host share one buffer (one device-to-host copy)
        self._out_pack, outs = _packed(dict(out_tokens=torch.empty((Bn, w.max_path), dtype=torch.int32),
                                            out_len=torch.empty(Bn, dtype=torch.int32),
                                            new_kv_len=torch.empty(Bn, dtype=torch.int32)), dev)
        self.out_tokens, self.out_len = outs["out_tokens"], outs["out_len"]
        self.path = torch.empty((Bn, w.max_path), **i32)
        self.n_acc = torch.empty(Bn, **i32)
        self.rejections = torch.empty(Bn, **i32)
        self.new_kv_len = outs["new_kv_len"]
        self._in_pack = None   # set by twin(): the per-round inputs in one device buffer
        self.blocks_in_use = torch.empty(Bn, **i32)
        self.slot_map = torch.empty((Bn, w.max_path, 2), **i32)
        self.k_layer0 = w.k_cache[0]
        self.v_layer0 = w.v_cache[0]
        self.attn = B.attention_params(w.q, self.k_layer0, self.v_layer0, w.block_table,
                                       w.prefix_len, w.node_offset, self.anc_mask, w.T_max,
                                       self.o, self.lse, self.req_status)
        self.attn_ws = _ws(B.spec_attention_workspace_size(self.attn), dev)
        self.ver = B.verify_params(w.target, w.draft, w.draft_kind, w.draft_row, w.tokens,
                                   w.parent, w.node_offset, self.depth, self.is_internal,
                                   w.uniforms, w.tau, w.V, w.T_max, w.max_path, self.req_status,
                                   self.out_tokens, self.out_len, self.path, self.n_acc,
                                   self.rejections, sibling_rule, verify_path)
        self.ver_ws = _ws(B.spec_verify_workspace_size(self.ver), dev)
        self.comp = B.compact_params(w.k_cache, w.v_cache, w.block_table, w.prefix_len,
                                     self.path, self.n_acc, self.req_status, self.new_kv_len,
                                     self.slot_map, self.blocks_in_use, w.max_path)
        self.rope_p = None

    def enable_rope(self, q_raw, k_new, v_new, base=10000.0, rotary_dim=None, interleaved=False,
                    fused=True):
        """Add the step before attention to every round: q_raw, k_new, v_new ([N, H, d], the
        tree tokens' projections before position encoding) are rotated at the tree's position
        ids into the workload's q and into the tree slots of layer 0's cache.  fused: run it
        inside the tree build's launch (spec_tree_build_rope_kv_write) instead of as a call of
        its own after it."""
        w = self.w
        self.rope_fused = fused
        self.rope_inputs = (q_raw, k_new, v_new)
        self.rope_p = B.rope_params(q_raw, w.q, k_new, v_new, self.k_layer0, self.v_layer0,
                                    w.block_table, w.prefix_len, w.node_offset, self.pos_id,
                                    self.req_status, base, rotary_dim, interleaved)

    # individual stages ---------------------------------------------------------------------
    def tree_build_rope(self, stream=None):
        w = self.w
        B.spec_tree_build_rope_kv_write(w.parent, w.node_offset, w.prefix_len, w.T_max,
                                        self.depth, self.pos_id, self.anc_mask,
                                        self.is_internal, self.req_status, self.rope_p, stream)

    def tree_build(self, stream=None):
        w = self.w
        B.spec_tree_build(w.parent, w.node_offset, w.prefix_len, w.T_max, self.depth, self.pos_id,
                          self.anc_mask, self.is_internal, self.req_status, stream)

    def rope(self, stream=None):
        B.spec_tree_rope_kv_write(self.rope_p, stream)

    def attention(self, stream=None):
        B.spec_tree_attention(self.attn, self.attn_ws, stream)

    def verify(self, stream=None):
        B.spec_verify(self.ver, self.ver_ws, stream)

    def compact(self, stream=None):
        B.spec_kv_compact(self.comp, stream)

    def verify_compact(self, stream=None):
        """verify() then compact() as one call (spec_verify_compact: one kernel for both when
        the verification takes its one-launch form)."""
        B.spec_verify_compact(self.ver, self.comp, self.ver_ws, stream)

    def run(self, stream=None):
        """One full round: tree build, attention, then verification and compaction as one call
        (1 + 2 + 1 kernel launches on the stream; for trees of more than 32 nodes the
        verification and compaction take 1 + 1 launches in the walk form, the default from a
        vocabulary of 65536, and 2 + 1 in the two-launch form); with enable_rope, the tree build and
        the rotary step share one launch, or run as two calls when fused=False."""
        if self.rope_p is not None and self.rope_fused:
            self.tree_build_rope(stream)
        else:
            self.tree_build(stream)
            if self.rope_p is not None:
                self.rope(stream)
        self.attention(stream)
        self.verify_compact(stream)

    def capture_graph(self) -> "torch.cuda.CUDAGraph":
        """One round (run()) captured as a CUDA graph; replay() re-runs it on the same buffers.
        The launches keep their programmatic dependencies inside the graph.  Call run() once
        before capturing (first calls set per-device kernel attributes, which capture does not
        allow)."""
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                self.run(side)
        torch.cuda.current_stream().wait_stream(side)
        return g

    def results(self) -> Dict[str, torch.Tensor]:
        return dict(req_status=self.req_status, depth=self.depth, pos_id=self.pos_id,
                    anc_mask=self.anc_mask, is_internal=self.is_internal, o=self.o, lse=self.lse,
                    out_tokens=self.out_tokens, out_len=self.out_len, path=self.path,
                    n_acc=self.n_acc, rejections=self.rejections, new_kv_len=self.new_kv_len,
                    slot_map=self.slot_map, blocks_in_use=self.blocks_in_use)

    # end-to-end form ----------------------------------------------------------------------
    def step_input_tensors(self) -> Dict[str, torch.Tensor]:
        """Device tensors that a new round brings from the host: the draft tree, its logits,
        uniforms, Q and the tree tokens' K/V rows (slots P..P+T-1 are written by the caller;
        here the whole layer-0 tree region is represented by the block-table-addressed cache
        rows, which stay resident) -- see run_from_host."""
        w = self.w
        return dict(parent=w.parent, node_offset=w.node_offset, prefix_len=w.prefix_len,
                    tokens=w.tokens, draft_row=w.draft_row, uniforms=w.uniforms, target=w.target,
                    draft=w.draft, q=w.q, block_table=w.block_table)

    def pinned_host_inputs(self) -> Dict[str, torch.Tensor]:
        """The round's inputs in pinned host memory: one packed buffer ("_pack", same layout as
        the step's device pack) for a step made by twin(), else one tensor per input."""
        if self._in_pack is not None:
            host = torch.empty(self._in_pack.numel(), dtype=torch.uint8).pin_memory()
            host.copy_(self._in_pack)
            return {"_pack": host}
        return {k: v.detach().to("cpu").pin_memory() for k, v in self.step_input_tensors().items()}

    def upload(self, host_inputs: Dict[str, torch.Tensor], stream=None):
        """Copy a round's inputs from pinned host memory to this step's device tensors, on
        `stream` (default: the current stream)."""
        with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream()):
            if "_pack" in host_inputs:
                if self._in_pack is None or self._in_pack.numel() != host_inputs["_pack"].numel():
                    raise ValueError("a packed upload needs a step made by twin() of the same shape")
                self._in_pack.copy_(host_inputs["_pack"], non_blocking=True)
                return
            dev_in = self.step_input_tensors()
            for k, h in host_inputs.items():
                dev_in[k].copy_(h, non_blocking=True)

    def download(self, host_out: Dict[str, torch.Tensor], stream=None):
        """Copy the accepted tokens, lengths and new KV lengths to pinned host memory."""
        with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream()):
            host_out["_pack"].copy_(self._out_pack, non_blocking=True)

    def run_from_host(self, host_inputs: Dict[str, torch.Tensor], host_out: Dict[str, torch.Tensor],
                      stream=None):
        """Copy the round's inputs from pinned host memory, run the round, copy the accepted
        tokens and lengths back.  Asynchronous on the stream; synchronise before reading
        host_out."""
        self.upload(host_inputs, stream)
        self.run(stream)
        self.download(host_out, stream)

    def twin(self) -> "VerifyStep":
        """A second step of the same shape over its own copies of the per-round input tensors
        and the same KV cache: while one step runs a round, the next round's inputs can be
        uploaded into the other (double buffering)."""
        src = self.step_input_tensors()
        pack, fresh = _packed(src, self.w.target.device)
        for k, v in fresh.items():
            v.copy_(src[k])
        step = VerifyStep(dataclasses.replace(self.w, **fresh), self.sibling_rule,
                          self.lse is not None, self.verify_path)
        step._in_pack = pack
        return step

    def host_output_buffers(self) -> Dict[str, torch.Tensor]:
        """Pinned host buffers for download(): "_pack" and the views out_tokens, out_len,
        new_kv_len into it."""
        pack, views = _packed(dict(out_tokens=self.out_tokens, out_len=self.out_len,
                                   new_kv_len=self.new_kv_len), "cpu", pin=True)
        return {"_pack": pack, **views}

    @staticmethod
    def bytes_of(tensors: Dict[str, torch.Tensor]) -> int:
        """Bytes one copy of these buffers moves (a packed buffer counts once, padding included)."""
        if "_pack" in tensors:
            return tensors["_pack"].numel() * tensors["_pack"].element_size()
        return sum(t.numel() * t.element_size() for t in tensors.values())


class RoundPipeline:
    """Rounds of one workload shape submitted from pinned host memory, double-buffered.

    Two twins of a step (own input and output buffers, the same KV cache) alternate.  Each
    submit() enqueues: the round's upload on an upload stream, its kernels on the compute stream,
    and the read-back of its results on a download stream, ordered by events so that no copy sits
    between two rounds' kernels: round i's upload waits for round i - 2 (the last reader of that
    input buffer), round i's kernels wait for their inputs and for round i - 2's download (the
    same output buffer).  Everything is asynchronous; results of round i are in
    host_outputs(i) once finish() (or a later synchronisation) has returned."""

    def __init__(self, step: VerifyStep, stream=None):
        self.steps = [step.twin(), step.twin()]
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        self.up, self.dl = torch.cuda.Stream(), torch.cuda.Stream()
        self.ready = [torch.cuda.Event(), torch.cuda.Event()]
        self.done = [torch.cuda.Event(), torch.cuda.Event()]
        self.dl_done = [torch.cuda.Event(), torch.cuda.Event()]
        self.host_outs = [step.host_output_buffers(), step.host_output_buffers()]
        for k in range(2):
            self.done[k].record(self.stream)
            self.dl_done[k].record(self.stream)
        self.up.wait_stream(self.stream)
        self.dl.wait_stream(self.stream)
        self.count = 0

    def pinned_host_inputs(self) -> Dict[str, torch.Tensor]:
        """A pinned host buffer in the layout submit() takes."""
        return self.steps[0].pinned_host_inputs()

    def host_outputs(self, i: int) -> Dict[str, torch.Tensor]:
        """The pinned host results of round i (valid until round i + 2 is submitted)."""
        return self.host_outs[i % 2]

    def submit(self, host_inputs: Dict[str, torch.Tensor]) -> int:
        k = self.count % 2
        st = self.steps[k]
        self.up.wait_event(self.done[k])
        st.upload(host_inputs, self.up)
        self.ready[k].record(self.up)
        self.stream.wait_event(self.ready[k])
        self.stream.wait_event(self.dl_done[k])
        st.run(self.stream)
        self.done[k].record(self.stream)
        self.dl.wait_event(self.done[k])
        st.download(self.host_outs[k], self.dl)
        self.dl_done[k].record(self.dl)
        self.count += 1
        return self.count - 1

    def finish(self):
        """Make the compute stream wait for every submitted round's results on the host."""
        self.stream.wait_stream(self.dl)


class DraftTreeBuilder:
    """The device side of building a draft tree for a batch: EAGLE-2 expansion of the K most
    probable leaves per level, the K most probable tokens of each expanded row, and ECHO's
    batch-wide budget of K_max tokens, packed for verification.  The draft model's forward
    (candidates -> draft rows) is the caller's: between expand(level) and append(level, rows)
    it writes row r * K + j of `rows` for the candidate expand_list[r, j].

    Owns the candidate pool (capacity `cap` per request), the expand list, the ECHO workspace
    and the packed outputs; every call is asynchronous on the current stream."""

    def __init__(self, batch: int, K: int, depth: int, device, cap: Optional[int] = None):
        cap = cap if cap is not None else 1 + K + (depth - 1) * K * K
        if cap > B.SPEC_MAX_TREE:
            raise ValueError(f"pool capacity above {B.SPEC_MAX_TREE} candidates per request")
        self.B, self.K, self.depth, self.cap = batch, K, depth, cap
        nb = batch
        i32 = dict(dtype=torch.int32, device=device)
        self.parent = torch.full((nb, cap), -1, **i32)
        self.token = torch.zeros((nb, cap), **i32)
        self.depth_ = torch.zeros((nb, cap), **i32)
        self.score = torch.zeros((nb, cap), dtype=torch.float32, device=device)
        self.row = torch.full((nb, cap), -1, **i32)
        self.count = torch.zeros(nb, **i32)
        self.req_status = torch.zeros(nb, **i32)
        self.expand_list = torch.full((nb, K), -1, **i32)
        self.pool = _pool(self)
        self.echo_ws = _ws(B.spec_echo_workspace_size(nb, cap), device)
        n = nb * cap
        self.node_offset = torch.zeros(nb + 1, **i32)
        self.tree_parent = torch.zeros(n, **i32)
        self.tree_tokens = torch.zeros(n, **i32)
        self.tree_depth = torch.zeros(n, **i32)
        self.tree_draft_row = torch.zeros(n, **i32)
        self.tree_source = torch.zeros(n, **i32)

    def init(self, root_tokens: torch.Tensor, stream=None):
        self.req_status.zero_()
        B.spec_draft_init(self.pool, root_tokens, stream)

    def expand(self, level: int, stream=None):
        B.spec_draft_expand_select(self.pool, level, self.K, self.expand_list, self.req_status,
                                    stream)

    def append(self, level: int, rows: torch.Tensor, V: int, tau: float = 1.0, stream=None):
        """rows: [B * K, ld] draft logits of the listed candidates (level's rows numbered
        (level - 1) * B * K + r * K + j in the packed draft_row)."""
        B.spec_draft_topk_append(self.pool, level, self.K, self.expand_list, rows, V, tau,
                                  (level - 1) * self.B * self.K, self.req_status, stream)

    def echo(self, K_max: int, stream=None):
        B.spec_echo_select_pack(self.pool, K_max, self.node_offset, self.tree_parent,
                                 self.tree_tokens, self.tree_depth, self.tree_draft_row,
                                 self.tree_source, self.echo_ws, stream)

    def packed(self) -> Dict[str, torch.Tensor]:
        """The packed trees (synchronises to read N)."""
        N = int(self.node_offset[-1])
        return dict(node_offset=self.node_offset, parent=self.tree_parent[:N],
                    tokens=self.tree_tokens[:N], depth=self.tree_depth[:N],
                    draft_row=self.tree_draft_row[:N], source=self.tree_source[:N])


def _pool(b: "DraftTreeBuilder"):
    return B.draft_pool(b.parent, b.token, b.depth_, b.score, b.row, b.count)
