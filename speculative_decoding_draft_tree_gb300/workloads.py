"""Seeded synthetic inputs for the draft-tree verification step.

This module only *generates inputs*: draft-tree shapes, target and draft logits, Q and the
paged K/V cache, block tables, prefix lengths and the explicit per-node uniforms the ratio test
consumes.  It holds none of the verification arithmetic (no tree mask, no attention, no ratio
test, no residual sampling, no compaction); both the CUDA library and the CPU oracle take what
it produces as plain inputs.  Drafting-side choices (which tokens a draft model proposes, which
tree an EAGLE-2/ECHO drafter would keep) are made here with library routines (softmax, top-k,
multinomial) because drafting is outside the verified path.

Sources of the shapes (page title, section):
  * chain drafts and the ratio test: "推测解码 2026" (guijiagi.com), 数学基础：拒绝采样;
  * Medusa Cartesian tree 3/5/7 -> 3 + 3*5 + 3*5*7 = 123 drafts: "万字综述 10+ 种 LLM 投机采样推理加速方案"
    (m.haoling.cc), section 6.2;
  * SpecInfer expansion tree with K = 3,2,2,1,1 -> 45 drafts, EAGLE-2 top-K leaf expansion by
    cumulative path probability, ECHO global verify budget K_max: "投机推理算法的常见优化手段"
    (cnblogs zrq96), 草稿树的生成 and 动态草稿长度.

Uniforms are Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
1, 2, 3", SC'11), key = (seed, 0), counter = (global node id, round, 0, 0); output word 0 is the
node's acceptance uniform and word 1 its sampling uniform, each mapped to [0, 1) as
(x >> 8) * 2^-24 so that it is exact in fp32 and fp64 alike.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

# ----------------------------------------------------------------------------------------------
# Philox4x32-10 (SC'11): two 32x32->64 multiplies per round, Weyl key schedule.
# ----------------------------------------------------------------------------------------------
_PHILOX_M0 = np.uint64(0xD2511F53)
_PHILOX_M1 = np.uint64(0xCD9E8D57)
_PHILOX_W0 = np.uint64(0x9E3779B9)
_PHILOX_W1 = np.uint64(0xBB67AE85)
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(counters: np.ndarray, key: Sequence[int]) -> np.ndarray:
    """Philox4x32 with 10 rounds.  counters: uint32 [n, 4]; key: two uint32 words.

    Returns uint32 [n, 4].  Each round multiplies counter words 0 and 2 by the two Philox
    constants, mixes the high halves with words 1 and 3 and the key, and the key is bumped by
    the Weyl increments between rounds.
    """
    c = np.asarray(counters, dtype=np.uint64).reshape(-1, 4)
    c0, c1, c2, c3 = c[:, 0].copy(), c[:, 1].copy(), c[:, 2].copy(), c[:, 3].copy()
    k0 = np.uint64(int(key[0]) & 0xFFFFFFFF)
    k1 = np.uint64(int(key[1]) & 0xFFFFFFFF)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + _PHILOX_W0) & _MASK32
            k1 = (k1 + _PHILOX_W1) & _MASK32
        p0 = _PHILOX_M0 * c0
        p1 = _PHILOX_M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0) & _MASK32, lo1, (hi0 ^ c3 ^ k1) & _MASK32, lo0
    return np.stack([c0, c1, c2, c3], axis=1).astype(np.uint32)


def node_uniforms(num_nodes: int, seed: int = 0, round_id: int = 0,
                  first_node: int = 0) -> np.ndarray:
    """float32 [num_nodes, 2]: (u_acc, u_samp) for global node ids first_node.. ."""
    ctr = np.zeros((num_nodes, 4), dtype=np.uint64)
    ctr[:, 0] = np.arange(first_node, first_node + num_nodes, dtype=np.uint64)
    ctr[:, 1] = round_id
    out = philox4x32_10(ctr, (seed, 0))
    u = (out[:, :2] >> np.uint32(8)).astype(np.float64) * (2.0 ** -24)
    return u.astype(np.float32)


# ----------------------------------------------------------------------------------------------
# Tree shapes (parent arrays in BFS order, root = node 0 with parent -1).
# ----------------------------------------------------------------------------------------------
def chain_parents(num_nodes: int) -> List[int]:
    """A chain root -> d1 -> d2 ...: num_nodes includes the root."""
    return [-1] + list(range(num_nodes - 1))


def cartesian_tree(ks: Sequence[int]):
    """Medusa Cartesian tree: every node on level l gets ks[l] children (BFS order).

    Returns (parents, levels); levels[i] is the construction level of node i."""
    parents, levels = [-1], [0]
    level = [0]
    for lvl, k in enumerate(ks):
        nxt = []
        for p in level:
            for _ in range(k):
                parents.append(p)
                levels.append(lvl + 1)
                nxt.append(len(parents) - 1)
        level = nxt
    return parents, levels


def cartesian_parents(ks: Sequence[int]) -> List[int]:
    return cartesian_tree(ks)[0]


def expansion_parents(schedule: Sequence[int]) -> List[int]:
    """SpecInfer expansion tree: each node at depth l gets schedule[l] children."""
    return cartesian_parents(schedule)


# ----------------------------------------------------------------------------------------------
# Workload container.
# ----------------------------------------------------------------------------------------------
DRAFT_LOGITS = 0
DRAFT_PROBS = 1
SIBLING_RESIDUAL = 0
SIBLING_INDEPENDENT = 1


@dataclass
class Workload:
    name: str
    dtype: str                 # "f32" or "bf16": logits, Q, K/V and O element type
    B: int
    V: int                     # vocabulary size (columns that are meaningful)
    H_q: int
    H_kv: int
    d: int
    bs: int                    # KV block size (tokens per block)
    tau: float
    draft_kind: int
    T_max: int
    max_path: int
    node_offset: torch.Tensor  # int32 [B+1]
    parent: torch.Tensor       # int32 [N], local index of the parent, -1 for the root
    tokens: torch.Tensor       # int32 [N]
    draft_row: torch.Tensor    # int32 [N], draft row holding q for node i's children, -1 if none
    prefix_len: torch.Tensor   # int32 [B]
    target: torch.Tensor       # [N, ld] logits (dtype), first V columns meaningful
    draft: torch.Tensor        # [R, ld] draft logits (dtype) or probabilities (fp32)
    uniforms: torch.Tensor     # fp32 [N, 2]
    q: torch.Tensor            # [N, H_q, d]
    k_cache: torch.Tensor      # [L, num_blocks, H_kv, bs, d]
    v_cache: torch.Tensor      # [L, num_blocks, H_kv, bs, d]
    block_table: torch.Tensor  # int32 [B, max_blocks]
    meta: Dict = field(default_factory=dict)

    @property
    def N(self) -> int:
        return int(self.node_offset[-1])

    @property
    def R(self) -> int:
        return int(self.draft.shape[0])

    @property
    def num_layers(self) -> int:
        return int(self.k_cache.shape[0])

    def tree_sizes(self) -> List[int]:
        no = self.node_offset.cpu().tolist()
        return [no[i + 1] - no[i] for i in range(self.B)]

    def to(self, device) -> "Workload":
        kw = {}
        for f in self.__dataclass_fields__:
            v = getattr(self, f)
            kw[f] = v.to(device) if isinstance(v, torch.Tensor) else v
        return Workload(**kw)


def _torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _row_ld(V: int, dtype: str) -> int:
    """Row stride in elements: rows start on 16-byte boundaries."""
    per16 = 16 // (4 if dtype == "f32" else 2)
    return (V + per16 - 1) // per16 * per16


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _pad_rows(x: torch.Tensor, ld: int) -> torch.Tensor:
    if x.shape[1] == ld:
        return x.contiguous()
    out = torch.zeros(x.shape[0], ld, dtype=x.dtype, device=x.device)
    out[:, : x.shape[1]] = x
    return out


def _paged_cache(B: int, kv_slots: Sequence[int], H_kv: int, d: int, bs: int, dtype: str,
                 device, num_layers: int, contiguous: bool, seed_qkv: int, seed_perm: int,
                 slack: float = 0.10):
    """Random K/V pool plus a block table covering kv_slots[r] logical slots per request."""
    need = [max(1, math.ceil(s / bs)) for s in kv_slots]
    max_blocks = max(need)
    if contiguous:
        num_blocks = B * max_blocks
        table = np.full((B, max_blocks), -1, dtype=np.int32)
        for r in range(B):
            table[r, : need[r]] = r * max_blocks + np.arange(need[r])
    else:
        total = sum(need)
        num_blocks = total + max(1, int(math.ceil(total * slack)))
        perm = np.random.default_rng(seed_perm).permutation(num_blocks).astype(np.int32)
        table = np.full((B, max_blocks), -1, dtype=np.int32)
        pos = 0
        for r in range(B):
            table[r, : need[r]] = perm[pos: pos + need[r]]
            pos += need[r]
    g = _gen(seed_qkv + 17, device)
    shape = (num_layers, num_blocks, H_kv, bs, d)
    td = _torch_dtype(dtype)
    k = torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(td)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(td)
    return k, v, torch.from_numpy(table).to(device)


def _finish(name, dtype, B, V, H_q, H_kv, d, bs, tau, parents_per_req, tokens, draft_row,
            prefix, target, draft, device, num_layers, contiguous, seeds, T_max=None,
            draft_kind=DRAFT_LOGITS, meta=None) -> Workload:
    sizes = [len(p) for p in parents_per_req]
    node_offset = np.zeros(B + 1, dtype=np.int32)
    node_offset[1:] = np.cumsum(sizes)
    N = int(node_offset[-1])
    parent = np.concatenate([np.asarray(p, dtype=np.int32) for p in parents_per_req])
    T_max = T_max if T_max is not None else max(sizes)
    ld = _row_ld(V, dtype if draft_kind == DRAFT_LOGITS else "f32")
    td = _torch_dtype(dtype)
    target = _pad_rows(target.to(td), _row_ld(V, dtype))
    if draft_kind == DRAFT_LOGITS:
        draft = _pad_rows(draft.to(td), ld)
    else:
        draft = _pad_rows(draft.to(torch.float32), _row_ld(V, "f32"))
    gq = _gen(seeds["qkv"], device)
    q = torch.randn((N, H_q, d), generator=gq, device=device, dtype=torch.float32).to(td)
    kv_slots = [int(prefix[r]) + sizes[r] for r in range(B)]
    k, v, table = _paged_cache(B, kv_slots, H_kv, d, bs, dtype, device, num_layers, contiguous,
                               seeds["qkv"], seeds["perm"])
    u = node_uniforms(N, seed=seeds["uniform"])
    return Workload(
        name=name, dtype=dtype, B=B, V=V, H_q=H_q, H_kv=H_kv, d=d, bs=bs, tau=float(tau),
        draft_kind=draft_kind, T_max=int(T_max), max_path=int(T_max),
        node_offset=torch.from_numpy(node_offset).to(device),
        parent=torch.from_numpy(parent).to(device),
        tokens=torch.as_tensor(np.asarray(tokens, dtype=np.int32)).to(device),
        draft_row=torch.as_tensor(np.asarray(draft_row, dtype=np.int32)).to(device),
        prefix_len=torch.as_tensor(np.asarray(prefix, dtype=np.int32)).to(device),
        target=target, draft=draft, uniforms=torch.from_numpy(u).to(device), q=q,
        k_cache=k, v_cache=v, block_table=table, meta=dict(meta or {}))


SEEDS = dict(logits=1, drafting=2, qkv=3, kvlen=4, perm=5, uniform=0)


def new_tree_kv(w: "Workload", seed: int = SEEDS["qkv"] + 29):
    """The tree tokens' own K and V rows before they enter the cache: N(0, 1) in the workload's
    dtype, [N, H_kv, d] each, on the workload's device (inputs of the RoPE + K/V write step)."""
    g = _gen(seed, w.q.device)
    shape = (w.N, w.H_kv, w.d)
    td = _torch_dtype(w.dtype)
    k = torch.randn(shape, generator=g, device=w.q.device, dtype=torch.float32).to(td)
    v = torch.randn(shape, generator=g, device=w.q.device, dtype=torch.float32).to(td)
    return k, v


# ----------------------------------------------------------------------------------------------
# Chains (configurations 1 and 2).
# ----------------------------------------------------------------------------------------------
def chain_workload(*, B: int, gamma: int, V: int, dtype: str, H_q: int, H_kv: int, d: int,
                   prefix, tau: float, target_std: float, noise_std: float, device="cpu",
                   bs: int = 16, num_layers: int = 1, contiguous: bool = False,
                   draft_kind: int = DRAFT_LOGITS, name: str = "chain",
                   seeds: Optional[Dict] = None, T_max: Optional[int] = None) -> Workload:
    """B chains of gamma drafts.  Each internal node i has its own draft row
    draft_i = target_i + N(0, noise_std^2); node i+1's token is drawn from softmax(draft_i)
    (tau > 0) or is argmax(draft_i) (tau == 0)."""
    seeds = dict(SEEDS, **(seeds or {}))
    T = gamma + 1
    g = _gen(seeds["logits"], device)
    tgt = torch.randn((B * T, V), generator=g, device=device) * target_std
    internal = [r * T + i for r in range(B) for i in range(gamma)]
    drf = tgt[internal] + torch.randn((len(internal), V), generator=g, device=device) * noise_std
    gd = _gen(seeds["drafting"], device)
    if tau > 0:
        probs = torch.softmax(drf.to(_torch_dtype(dtype)).float(), dim=-1)
        picks = torch.multinomial(probs, 1, generator=gd).squeeze(1)
    else:
        picks = drf.to(_torch_dtype(dtype)).float().argmax(dim=-1)
    picks = picks.cpu().numpy()
    roots = torch.randint(0, V, (B,), generator=gd, device=device).cpu().numpy()
    tokens = np.zeros(B * T, dtype=np.int32)
    draft_row = np.full(B * T, -1, dtype=np.int32)
    for r in range(B):
        tokens[r * T] = roots[r]
        for i in range(gamma):
            tokens[r * T + i + 1] = picks[r * gamma + i]
            draft_row[r * T + i] = r * gamma + i
    if draft_kind == DRAFT_PROBS:
        # the drafter hands over the distribution it sampled from (temperature 1)
        drf = torch.softmax(drf.to(_torch_dtype(dtype)).float(), dim=-1)
    prefix = list(prefix) if hasattr(prefix, "__len__") else [int(prefix)] * B
    return _finish(name, dtype, B, V, H_q, H_kv, d, bs, tau, [chain_parents(T)] * B, tokens,
                   draft_row, prefix, tgt, drf, device, num_layers, contiguous, seeds,
                   T_max=T_max, draft_kind=draft_kind,
                   meta=dict(kind="chain", gamma=gamma, noise_std=noise_std))


# ----------------------------------------------------------------------------------------------
# Static trees whose children are the top-k of a draft row (configurations 3 and 4).
# ----------------------------------------------------------------------------------------------
def _topk_children_tokens(rows: torch.Tensor, k: int) -> np.ndarray:
    return torch.topk(rows.float(), k, dim=-1).indices.cpu().numpy().astype(np.int32)


def medusa_workload(*, B: int, ks=(3, 5, 7), V: int, dtype: str, H_q: int, H_kv: int, d: int,
                    prefix, tau: float, target_std: float = 3.0, noise_std: float = 1.0,
                    device="cpu", bs: int = 16, num_layers: int = 1,
                    seeds: Optional[Dict] = None, name: str = "medusa",
                    T_max: Optional[int] = None) -> Workload:
    """Medusa Cartesian tree.  Head l (l = 1..len(ks)) proposes the top-ks[l-1] tokens of its
    row; the row is the target row of the first node at depth l-1 plus N(0, noise_std^2).
    Every node at depth l-1 shares head l's row (draft_row) and candidate tokens."""
    seeds = dict(SEEDS, **(seeds or {}))
    parents, depth = cartesian_tree(ks)
    T = len(parents)
    first_at_depth = [depth.index(l) for l in range(len(ks))]
    g = _gen(seeds["logits"], device)
    tgt = torch.randn((B * T, V), generator=g, device=device) * target_std
    heads = []
    for r in range(B):
        for l in range(len(ks)):
            heads.append(tgt[r * T + first_at_depth[l]]
                         + torch.randn((V,), generator=g, device=device) * noise_std)
    drf = torch.stack(heads)
    td = _torch_dtype(dtype)
    gd = _gen(seeds["drafting"], device)
    roots = torch.randint(0, V, (B,), generator=gd, device=device).cpu().numpy()
    tokens = np.zeros(B * T, dtype=np.int32)
    draft_row = np.full(B * T, -1, dtype=np.int32)
    for r in range(B):
        cand = [_topk_children_tokens(drf[r * len(ks) + l: r * len(ks) + l + 1].to(td), ks[l])[0]
                for l in range(len(ks))]
        tokens[r * T] = roots[r]
        child_rank = {}
        for i in range(1, T):
            p = parents[i]
            rank = child_rank.get(p, 0)
            child_rank[p] = rank + 1
            tokens[r * T + i] = cand[depth[p]][rank]
        for i in range(T):
            if depth[i] < len(ks):
                draft_row[r * T + i] = r * len(ks) + depth[i]
    prefix = list(prefix) if hasattr(prefix, "__len__") else [int(prefix)] * B
    return _finish(name, dtype, B, V, H_q, H_kv, d, bs, tau, [parents] * B, tokens, draft_row,
                   prefix, tgt, drf, device, num_layers, False, seeds, T_max=T_max,
                   meta=dict(kind="medusa", ks=tuple(ks)))


def specinfer_workload(*, B: int, schedule=(3, 2, 2, 1, 1), V: int, dtype: str, H_q: int,
                       H_kv: int, d: int, prefix, tau: float, target_std: float = 3.0,
                       noise_std: float = 1.0, device="cpu", bs: int = 16, num_layers: int = 1,
                       seeds: Optional[Dict] = None, name: str = "specinfer",
                       T_max: Optional[int] = None) -> Workload:
    """SpecInfer expansion tree: node i's draft row is target_i + N(0, noise_std^2) and its
    children are the top-schedule[depth(i)] tokens of that row."""
    seeds = dict(SEEDS, **(seeds or {}))
    parents, depth = cartesian_tree(schedule)
    T = len(parents)
    internal_local = [i for i in range(T) if depth[i] < len(schedule)]
    g = _gen(seeds["logits"], device)
    tgt = torch.randn((B * T, V), generator=g, device=device) * target_std
    idx = [r * T + i for r in range(B) for i in internal_local]
    drf = tgt[idx] + torch.randn((len(idx), V), generator=g, device=device) * noise_std
    td = _torch_dtype(dtype)
    gd = _gen(seeds["drafting"], device)
    roots = torch.randint(0, V, (B,), generator=gd, device=device).cpu().numpy()
    kmax = max(schedule)
    top = _topk_children_tokens(drf.to(td), kmax)
    tokens = np.zeros(B * T, dtype=np.int32)
    draft_row = np.full(B * T, -1, dtype=np.int32)
    nint = len(internal_local)
    for r in range(B):
        tokens[r * T] = roots[r]
        row_of = {i: r * nint + j for j, i in enumerate(internal_local)}
        child_rank = {}
        for i in range(1, T):
            p = parents[i]
            rank = child_rank.get(p, 0)
            child_rank[p] = rank + 1
            tokens[r * T + i] = top[row_of[p], rank]
        for i in internal_local:
            draft_row[r * T + i] = row_of[i]
    prefix = list(prefix) if hasattr(prefix, "__len__") else [int(prefix)] * B
    return _finish(name, dtype, B, V, H_q, H_kv, d, bs, tau, [parents] * B, tokens, draft_row,
                   prefix, tgt, drf, device, num_layers, False, seeds, T_max=T_max,
                   meta=dict(kind="specinfer", schedule=tuple(schedule)))


# ----------------------------------------------------------------------------------------------
# EAGLE-2 dynamic trees under an ECHO global budget (configuration 5).
# ----------------------------------------------------------------------------------------------
def eagle2_echo_workload(*, B: int, V: int, dtype: str, H_q: int, H_kv: int, d: int,
                         prefix_range=(1024, 32768), tau: float = 1.0, topk: int = 5,
                         max_depth: int = 8, K_max: int = 2048, target_std: float = 3.0,
                         noise_std: float = 1.0, device="cpu", bs: int = 16, num_layers: int = 1,
                         seeds: Optional[Dict] = None, name: str = "eagle2_echo",
                         T_max: int = 256, prefix=None) -> Workload:
    """Dynamic ragged trees.  Level 1 expands the root; every later level expands only the
    top-`topk` nodes of the newest level by cumulative path probability (product of draft
    probabilities along the path), each into the top-`topk` tokens of its draft row
    (draft = target + N(0, noise_std^2)).  The batch then keeps the global top-K_max nodes by
    cumulative path probability (roots always kept; ties by request, then node index), which is
    closed under ancestors because a parent's cumulative probability is never below its
    child's."""
    seeds = dict(SEEDS, **(seeds or {}))
    g = _gen(seeds["logits"], device)
    gd = _gen(seeds["drafting"], device)
    td = _torch_dtype(dtype)
    # candidate nodes per request: (parent, token, depth, cum_logprob)
    roots = torch.randint(0, V, (B,), generator=gd, device=device).cpu().numpy()
    cand = [[(-1, int(roots[r]), 0, 0.0)] for r in range(B)]
    rows_t: Dict = {}   # (r, local) -> target row (fp32 tensor)
    rows_d: Dict = {}
    frontier = [[0] for _ in range(B)]
    for level in range(1, max_depth + 1):
        expand = []
        for r in range(B):
            fr = sorted(frontier[r], key=lambda i: (-cand[r][i][3], i))[:topk]
            expand.extend((r, i) for i in sorted(fr))
        if not expand:
            break
        t = torch.randn((len(expand), V), generator=g, device=device) * target_std
        dr = t + torch.randn((len(expand), V), generator=g, device=device) * noise_std
        dr_q = dr.to(td).float()
        logq = torch.log_softmax(dr_q, dim=-1)
        top = torch.topk(logq, topk, dim=-1)
        top_i = top.indices.cpu().numpy()
        top_v = top.values.double().cpu().numpy()
        new_frontier = [[] for _ in range(B)]
        for j, (r, i) in enumerate(expand):
            rows_t[(r, i)] = t[j]
            rows_d[(r, i)] = dr[j]
            for c in range(topk):
                cand[r].append((i, int(top_i[j, c]), level, cand[r][i][3] + float(top_v[j, c])))
                new_frontier[r].append(len(cand[r]) - 1)
        frontier = new_frontier
    # ECHO budget: global top-K_max by cumulative path log-probability.
    allnodes = [(r, i) for r in range(B) for i in range(len(cand[r]))]
    nonroot = [(r, i) for (r, i) in allnodes if i > 0]
    nonroot.sort(key=lambda ri: (-cand[ri[0]][ri[1]][3], ri[0], ri[1]))
    keep_n = max(0, K_max - B)
    kept = set((r, 0) for r in range(B)) | set(nonroot[:keep_n])
    parents_per_req, tokens, draft_row = [], [], []
    tgt_rows, drf_rows = [], []
    for r in range(B):
        local = sorted(i for i in range(len(cand[r])) if (r, i) in kept)
        remap = {old: new for new, old in enumerate(local)}
        par = []
        has_child = set()
        for old in local:
            p = cand[r][old][0]
            par.append(-1 if p < 0 else remap[p])
            if p >= 0:
                has_child.add(p)
        parents_per_req.append(par)
        for old in local:
            tokens.append(cand[r][old][1])
            if (r, old) not in rows_t:
                rows_t[(r, old)] = torch.randn((V,), generator=g, device=device) * target_std
            tgt_rows.append(rows_t[(r, old)])
            if old in has_child:
                draft_row.append(len(drf_rows))
                drf_rows.append(rows_d[(r, old)])
            else:
                draft_row.append(-1)
    tgt = torch.stack(tgt_rows)
    drf = torch.stack(drf_rows) if drf_rows else torch.zeros((1, V), device=device)
    rng = np.random.default_rng(seeds["kvlen"])
    if prefix is None:
        prefix = rng.integers(prefix_range[0], prefix_range[1] + 1, size=B).tolist()
    return _finish(name, dtype, B, V, H_q, H_kv, d, bs, tau, parents_per_req, tokens, draft_row,
                   prefix, tgt, drf, device, num_layers, False, seeds, T_max=T_max,
                   meta=dict(kind="eagle2_echo", topk=topk, max_depth=max_depth, K_max=K_max))


# ----------------------------------------------------------------------------------------------
# The five workloads, at full size ("full") and at a size the CPU oracle finishes in seconds
# while still spanning several attention tiles, vocab vectors and a ragged tail ("small").
# ----------------------------------------------------------------------------------------------
CONFIG_NAMES = {
    1: "chain_g4_v1000_f32",
    2: "leviathan_chain_b16_g5_v32000",
    3: "medusa_3x5x7_b4_v32000",
    4: "specinfer_32211_b32_v128256",
    5: "eagle2_echo_b64_kmax2048_v152064",
}


# ----------------------------------------------------------------------------------------------
# Draft-model output for building trees on the device: one level's rows.
# ----------------------------------------------------------------------------------------------
def draft_level_rows(*, B: int, K: int, V: int, level: int, dtype: str = "bf16", device="cpu",
                     seed: int = SEEDS["drafting"], scales=None) -> torch.Tensor:
    """[B * K, ld] draft logits standing in for the draft model's output at one level: row
    r * K + j ~ N(0, scales[r]^2) (a larger scale = a more confident request), seeded by
    (seed, level); rows padded to a 16-byte multiple."""
    g = _gen(seed * 1000 + level, device)
    sc = torch.as_tensor(list(scales) if scales is not None else [1.0] * B, dtype=torch.float32,
                         device=device)
    x = torch.randn((B * K, V), generator=g, device=device) * sc.repeat_interleave(K)[:, None]
    return _pad_rows(x.to(_torch_dtype(dtype)), _row_ld(V, dtype))


# ----------------------------------------------------------------------------------------------
# Several draft models (multi-draft verification: every sibling carries its own model's q).
# ----------------------------------------------------------------------------------------------
def multidraft_parents(k: int, gamma: int) -> List[int]:
    """k chains of gamma drafts hanging off the root, chain m after chain m - 1 in node order:
    the root's children come from k different draft models."""
    parents = [-1]
    for _ in range(k):
        prev = 0
        for _g in range(gamma):
            parents.append(prev)
            prev = len(parents) - 1
    return parents


def multidraft_workload(*, B: int, k: int, gamma: int, V: int, dtype: str, H_q: int, H_kv: int,
                        d: int, prefix, tau: float, target_std: float = 3.0,
                        noise_stds=None, device="cpu", bs: int = 16, num_layers: int = 1,
                        draft_kind: int = DRAFT_LOGITS, seeds: Optional[Dict] = None,
                        name: str = "multidraft", T_max: Optional[int] = None) -> Workload:
    """k draft models each sample a chain of gamma tokens.  Model m's distribution at a node is
    the target row there plus N(0, noise_stds[m]^2) (its own noise, so siblings at the root
    carry different q); the token of each child is drawn from its model's softmax(row / tau)
    (argmax at tau = 0), and draft row c holds the q child c was drawn from (the multi-draft
    sibling rule's indexing; the root's entry is -1)."""
    seeds = dict(SEEDS, **(seeds or {}))
    noise_stds = list(noise_stds or [0.5 + 0.5 * m for m in range(k)])
    parents = multidraft_parents(k, gamma)
    T = len(parents)
    g = _gen(seeds["logits"], device)
    tgt = torch.randn((B * T, V), generator=g, device=device) * target_std
    model_of = [-1] + [m for m in range(k) for _ in range(gamma)]
    # one draft row per non-root node: its model's row at its parent's context
    rows = []
    for r in range(B):
        for c in range(1, T):
            rows.append(tgt[r * T + parents[c]]
                        + torch.randn((V,), generator=g, device=device) * noise_stds[model_of[c]])
    drf = torch.stack(rows)
    td = _torch_dtype(dtype)
    gd = _gen(seeds["drafting"], device)
    if tau > 0:
        probs = torch.softmax(drf.to(td).float() / tau, dim=-1)
        picks = torch.multinomial(probs, 1, generator=gd).squeeze(1)
    else:
        picks = drf.to(td).float().argmax(dim=-1)
    picks = picks.cpu().numpy()
    roots = torch.randint(0, V, (B,), generator=gd, device=device).cpu().numpy()
    tokens = np.zeros(B * T, dtype=np.int32)
    draft_row = np.full(B * T, -1, dtype=np.int32)
    for r in range(B):
        tokens[r * T] = roots[r]
        for c in range(1, T):
            tokens[r * T + c] = picks[r * (T - 1) + c - 1]
            draft_row[r * T + c] = r * (T - 1) + c - 1
    if draft_kind == DRAFT_PROBS:
        drf = torch.softmax(drf.to(td).float() / (tau if tau > 0 else 1.0), dim=-1)
    prefix = list(prefix) if hasattr(prefix, "__len__") else [int(prefix)] * B
    return _finish(name, dtype, B, V, H_q, H_kv, d, bs, tau, [parents] * B, tokens, draft_row,
                   prefix, tgt, drf, device, num_layers, False, seeds, T_max=T_max,
                   draft_kind=draft_kind, meta=dict(kind="multidraft", k=k, gamma=gamma))


def multidraft_config(*, scale: str = "full", device="cpu", tau: float = 1.0,
                      draft_kind: int = DRAFT_LOGITS, seeds: Optional[Dict] = None,
                      num_layers: int = 1) -> Workload:
    """Full: 5 draft models x 3 tokens (a 16-token tree, the SpecInfer multi-model setting),
    16 requests, vocab 32000, LLaMA-7B attention (32 x d128 MHA), 2048 cached tokens.  Small:
    3 models x 2 tokens, 3 requests, odd sizes."""
    if scale == "full":
        return multidraft_workload(B=16, k=5, gamma=3, V=32000, dtype="bf16", H_q=32, H_kv=32,
                                   d=128, prefix=2048, tau=tau, device=device, seeds=seeds,
                                   draft_kind=draft_kind, num_layers=num_layers,
                                   name="multidraft_k5_g3_b16_v32000")
    return multidraft_workload(B=3, k=3, gamma=2, V=2999, dtype="bf16", H_q=4, H_kv=2, d=128,
                               prefix=[40, 301, 7], tau=tau, device=device, seeds=seeds,
                               draft_kind=draft_kind, num_layers=num_layers,
                               name="multidraft_k3_g2_b3_small")


# ----------------------------------------------------------------------------------------------
# Lookahead decoding: one forward over a 2-D Jacobi window and G candidate n-grams.
# ----------------------------------------------------------------------------------------------
def lookahead_parents(W: int, N: int, G: int) -> List[int]:
    """Shape of one lookahead-decoding forward as a parent array: the current token; the window
    (step 0 at positions 1 .. W-1, step l at positions l .. l+W-1, each token after the token
    one step and one position back); then G candidate n-gram chains of N - 1 tokens each."""
    index = {(0, 0): 0}
    parents = [-1]
    for p in range(1, W):
        index[(0, p)] = len(parents)
        parents.append(index[(0, p - 1)])
    for l in range(1, N - 1):
        for p in range(l, l + W):
            index[(l, p)] = len(parents)
            parents.append(index[(l - 1, p - 1)])
    for _ in range(G):
        prev = 0
        for _k in range(1, N):
            parents.append(prev)
            prev = len(parents) - 1
    return parents


def lookahead_workload(*, B: int, W: int, N: int, G: int, V: int, dtype: str, H_q: int, H_kv: int,
                       d: int, prefix, device="cpu", bs: int = 16, num_layers: int = 1,
                       target_std: float = 3.0, seeds: Optional[Dict] = None,
                       name: str = "lookahead", T_max: Optional[int] = None) -> Workload:
    """Greedy (tau = 0) lookahead decoding.  Window tokens are random guesses; candidate 0 of
    request r follows the target's greedy choices for r mod N tokens (a pool hit of that
    length), the other candidates are random.  Draft rows are the target rows (unused at
    tau = 0)."""
    seeds = dict(SEEDS, **(seeds or {}))
    parents = lookahead_parents(W, N, G)
    T = len(parents)
    g = _gen(seeds["logits"], device)
    tgt = torch.randn((B * T, V), generator=g, device=device) * target_std
    greedy = tgt.to(_torch_dtype(dtype)).float().argmax(dim=-1).cpu().numpy()
    gd = _gen(seeds["drafting"], device)
    tokens = torch.randint(0, V, (B * T,), generator=gd, device=device).cpu().numpy()
    tokens = tokens.astype(np.int32)
    first_candidate = T - G * (N - 1)
    for r in range(B):
        hits = min(r % N, N - 1) if G > 0 else 0
        prev = 0
        for k in range(1, hits + 1):
            node = first_candidate + k - 1
            tokens[r * T + node] = greedy[r * T + prev]
            prev = node
    has_child = set(parents[1:])
    draft_row = np.array([r * T + i if i in has_child else -1 for r in range(B) for i in range(T)],
                         dtype=np.int32)
    prefix = list(prefix) if hasattr(prefix, "__len__") else [int(prefix)] * B
    return _finish(name, dtype, B, V, H_q, H_kv, d, bs, 0.0, [parents] * B, tokens, draft_row,
                   prefix, tgt, tgt.clone(), device, num_layers, False, seeds, T_max=T_max,
                   meta=dict(kind="lookahead", W=W, N=N, G=G))


def lookahead_config(*, scale: str = "full", device="cpu", seeds: Optional[Dict] = None,
                     num_layers: int = 1) -> Workload:
    """Full: W = 15, N = 5, G = 15 (120 tokens per forward, the 7B setting's compute multiple),
    8 requests, LLaMA-2-7B attention (32 x d128 MHA), 2048 cached tokens, vocab 32000.  Small:
    the page's W = 5, N = 4, G = 5 example (30 tokens), 3 requests, odd sizes."""
    if scale == "full":
        return lookahead_workload(B=8, W=15, N=5, G=15, V=32000, dtype="bf16", H_q=32, H_kv=32,
                                  d=128, prefix=2048, device=device, seeds=seeds,
                                  num_layers=num_layers, name="lookahead_w15_n5_g15_b8_v32000")
    return lookahead_workload(B=3, W=5, N=4, G=5, V=3001, dtype="bf16", H_q=4, H_kv=2, d=128,
                              prefix=[301, 17, 160], device=device, seeds=seeds,
                              num_layers=num_layers, name="lookahead_w5_n4_g5_b3_small")


def make_config(cid: int, *, scale: str = "full", device="cpu", tau: Optional[float] = None,
                sigma: float = 1.0, num_layers: int = 1, seeds: Optional[Dict] = None,
                batch: Optional[int] = None) -> Workload:
    """Workload `cid` (1..5) at full size or small.  `batch` (full size only) keeps the shape of
    every request and takes fewer or more of them (the EAGLE-2 / ECHO budget scales with it)."""
    full = scale == "full"
    if batch is not None and full and cid in (2, 3, 4, 5):
        return _make_batch(cid, batch, device=device, tau=tau, sigma=sigma,
                           num_layers=num_layers, seeds=seeds)
    name = CONFIG_NAMES[cid] + ("" if full else "_small")
    if cid == 1:
        return chain_workload(B=1, gamma=4, V=1000, dtype="f32", H_q=4, H_kv=4, d=64,
                              prefix=128, tau=1.0 if tau is None else tau, target_std=2.0,
                              noise_std=1.0, device=device, num_layers=num_layers, name=name,
                              seeds=seeds)
    if cid == 2:
        return chain_workload(B=16 if full else 3, gamma=5, V=32000 if full else 4003,
                              dtype="bf16", H_q=32 if full else 4, H_kv=32 if full else 4,
                              d=128, prefix=2048 if full else 300,
                              tau=1.0 if tau is None else tau, target_std=3.0, noise_std=sigma,
                              device=device, num_layers=num_layers, contiguous=True, name=name,
                              seeds=seeds)
    if cid == 3:
        return medusa_workload(B=4 if full else 2, ks=(3, 5, 7), V=32000 if full else 3001,
                               dtype="bf16", H_q=40 if full else 3, H_kv=40 if full else 3,
                               d=128, prefix=4096 if full else 257,
                               tau=1.0 if tau is None else tau, device=device,
                               num_layers=num_layers, name=name, seeds=seeds)
    if cid == 4:
        return specinfer_workload(B=32 if full else 3, schedule=(3, 2, 2, 1, 1),
                                  V=128256 if full else 5003, dtype="bf16",
                                  H_q=32 if full else 8, H_kv=8 if full else 2, d=128,
                                  prefix=8192 if full else 271,
                                  tau=1.0 if tau is None else tau, device=device,
                                  num_layers=num_layers, name=name, seeds=seeds)
    if cid == 5:
        if full:
            return eagle2_echo_workload(B=64, V=152064, dtype="bf16", H_q=64, H_kv=8, d=128,
                                        prefix_range=(1024, 32768),
                                        tau=1.0 if tau is None else tau, K_max=2048,
                                        device=device, num_layers=num_layers, name=name,
                                        seeds=seeds)
        return eagle2_echo_workload(B=4, V=3011, dtype="bf16", H_q=16, H_kv=2, d=128,
                                    prefix_range=(1, 700), tau=1.0 if tau is None else tau,
                                    K_max=150, device=device, num_layers=num_layers, name=name,
                                    seeds=seeds)
    raise ValueError(f"unknown configuration {cid}")


def _make_batch(cid: int, B: int, *, device, tau, sigma, num_layers, seeds) -> Workload:
    name = f"{CONFIG_NAMES[cid]}_batch{B}"
    t = 1.0 if tau is None else tau
    if cid == 2:
        return chain_workload(B=B, gamma=5, V=32000, dtype="bf16", H_q=32, H_kv=32, d=128,
                              prefix=2048, tau=t, target_std=3.0, noise_std=sigma, device=device,
                              num_layers=num_layers, contiguous=True, name=name, seeds=seeds)
    if cid == 3:
        return medusa_workload(B=B, ks=(3, 5, 7), V=32000, dtype="bf16", H_q=40, H_kv=40, d=128,
                               prefix=4096, tau=t, device=device, num_layers=num_layers,
                               name=name, seeds=seeds)
    if cid == 4:
        return specinfer_workload(B=B, schedule=(3, 2, 2, 1, 1), V=128256, dtype="bf16", H_q=32,
                                  H_kv=8, d=128, prefix=8192, tau=t, device=device,
                                  num_layers=num_layers, name=name, seeds=seeds)
    return eagle2_echo_workload(B=B, V=152064, dtype="bf16", H_q=64, H_kv=8, d=128,
                                prefix_range=(1024, 32768), tau=t, K_max=2048 * B // 64,
                                device=device, num_layers=num_layers, name=name, seeds=seeds)
