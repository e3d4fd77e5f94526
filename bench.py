"""Benchmark of the draft-tree verification round on GB300.

A step = one pass of the whole hot path over one batch of synthetic requests:
spec_tree_build + spec_tree_attention (one layer) + spec_verify_compact (verification and KV
compaction), all through the C-ABI library.  The headline workload is the EAGLE-2 / ECHO one
(64 requests, dynamic trees of depth <= 8 under a batch budget of 2048 tree tokens, vocab
152064, GQA 64/8 x d128, paged KV with 1024..32768 cached tokens per request, bf16, tau = 1);
the four other workloads (chain gamma 4 fp32; Leviathan chain, 16 x (1 + 5), vocab 32000;
Medusa 3/5/7, 4 x 124; SpecInfer 3,2,2,1,1, 32 x 46, vocab 128256) are measured the same way
in the same run and reported under "configs".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload CID] [--configs 1,2,3,4]
                  [--impl reference]

Prints ONE JSON line (rank 0).  For every workload: `value` = verified tree tokens per second
over all ranks (median of the K timed steps, each replayed as one CUDA graph of the step's
launches, L2 flushed before each; max over ranks), with p10 / p90 of the step time;
`step_roofline` divides the whole step's algorithmic bytes by that time; `roofline` is the
tree-attention call's (the dominant kernel); `e2e` repeats the measurement through the public
RoundPipeline (VerifyStep.upload / run / download) with every round's inputs copied from pinned
host memory and its results copied back inside the timed region; `stats` are the method's own
numbers (acceptance rate, emitted tokens per request); `parity` compares the step's outputs
with the CPU oracle's on the whole batch and counts the near-boundary exemptions;
`cpu_baseline` times the oracle on the host cores, one core and all cores.  `alpha_sweep`
measures the acceptance rate on the Leviathan chain shape for draft noise sigma in
{0.5, 1, 2} and tau in {0, 1} against the closed form E[L] = (1 - a^(g+1)) / (1 - a).  `next`
measures the rows after the path: the step before attention (rotary embedding + tree K/V
write), the lookahead-decoding mask, multi-draft verification and the device-side draft-tree
construction.  `--impl reference` times the CPU oracle on a bounded sample instead.
"""
import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = 5
OTHER_CONFIGS = "1,2,3,4"
FLUSH_BYTES = 256 << 20
NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e, nominal (the measured copy bandwidth is `peak`)
BAND = 1e-6                # near-boundary exemption band of the verification's parity bar


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD,
                    help="the headline workload (1..5)")
    ap.add_argument("--configs", default=OTHER_CONFIGS,
                    help="workloads measured alongside the headline ('' for none)")
    ap.add_argument("--batch", type=int, default=None,
                    help="requests of the headline workload (same shape per request; default: "
                         "the workload's own batch)")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-next", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=5.0,
                    help="seconds of single-core oracle work per workload and leg")
    ap.add_argument("--clocks-csv", default=None,
                    help="keep the nvidia-smi samples taken during the timed region in this file")
    return ap.parse_args(argv)


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    kind="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, kind="fallback")


def percentile(xs, q):
    s = sorted(xs)
    if not s:
        return float("nan")
    k = (len(s) - 1) * q / 100.0
    lo, hi = int(math.floor(k)), int(math.ceil(k))
    return s[lo] + (s[hi] - s[lo]) * (k - lo)


def median(xs):
    return percentile(xs, 50)


def workload_description(w, cid):
    sizes = w.tree_sizes()
    P = w.prefix_len.cpu().tolist()
    return {
        "workload": w.name,
        "batch_requests": w.B,
        "tree_tokens_per_step": int(sum(sizes)),
        "drafts_per_step": int(sum(sizes) - w.B),
        "tree_tokens_per_request": (sizes[0] if len(set(sizes)) == 1
                                    else f"{min(sizes)}..{max(sizes)}"),
        "vocab": w.V,
        "heads": f"{w.H_q}q/{w.H_kv}kv x d{w.d}",
        "prefix_len": P[0] if len(set(P)) == 1 else f"{min(P)}..{max(P)}",
        "kv_block": w.bs,
        "tau": w.tau,
        "tree": w.meta.get("kind"),
        "l2": (f"flushed between timed steps: {FLUSH_BYTES >> 20} MB write, then a "
               f"{FLUSH_BYTES >> 20} MB read of another buffer (no step data and no dirty "
               f"lines left in L2)"),
    }


def recorded_traffic(workload_name):
    """DRAM bytes per launch of the tree-attention kernels on `workload_name` from the
    committed ncu captures, or None when there is none or the kernel sources changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "attention_traffic.json")
    try:
        recs = json.load(open(path))["records"]
    except Exception:
        return None
    for rec in recs:
        if rec.get("workload") != workload_name:
            continue
        try:
            h = hashlib.sha256()
            for src in rec["sources"]:
                h.update(open(os.path.join(ROOT, src), "rb").read())
            if h.hexdigest() != rec["sources_sha256"]:
                return None
            return rec["dram_bytes_read_per_launch"] + rec["dram_bytes_write_per_launch"]
        except Exception:
            return None
    return None


def rope_bytes(w):
    """Algorithmic bytes of the RoPE + tree K/V write step: every tree token's q, new k and new
    v row read once and written once (q to the attention input, k and v to their cache slot)."""
    es = 2 if w.dtype == "bf16" else 4
    return 2 * w.N * (w.H_q + 2 * w.H_kv) * w.d * es


def attention_bytes(w):
    """Algorithmic bytes of one tree-attention launch: each request's P + T keys of K and V for
    every KV head read once, Q read once, O and LSE written once."""
    es = 2 if w.dtype == "bf16" else 4
    sizes = w.tree_sizes()
    P = w.prefix_len.cpu().tolist()
    kv = sum((P[r] + sizes[r]) for r in range(w.B)) * w.H_kv * w.d * es * 2
    q_o = 2 * w.N * w.H_q * w.d * es
    return kv + q_o + w.N * w.H_q * 4


def attention_flops(w):
    """Tensor flops of one tree-attention launch: QK^T and PV over each node's visible keys
    (its request's prefix plus its own path), 2 flops per multiply-add, every query head."""
    import numpy as np
    no = w.node_offset.cpu().numpy()
    P = w.prefix_len.cpu().numpy()
    par = w.parent.cpu().numpy()
    total = 0
    for r in range(w.B):
        o, T = int(no[r]), int(no[r + 1] - no[r])
        depth = np.zeros(T, dtype=np.int64)
        for i in range(1, T):
            depth[i] = depth[par[o + i]] + 1
        total += int((P[r] + depth + 1).sum())
    return 4 * total * w.H_q * w.d


def step_bytes(w, step):
    """Algorithmic bytes of one whole step: the attention launch's, the verification's (every
    internal node's target row and every draft row an internal node names read once, plus one
    target and one draft row per request for the final draw) and the compaction's (K and V of
    every moved slot read and written, per layer); the tree build's few bytes per node are left
    out.  The moved slots are read from the step's own slot map after a round."""
    es = 2 if w.dtype == "bf16" else 4
    internal = step.is_internal.cpu().numpy().astype(bool)
    rows = int(internal.sum())
    drows = len(set(w.draft_row.cpu().numpy()[internal].tolist())) if w.tau > 0 else 0
    ver = (rows + drows + w.B * (2 if w.tau > 0 else 1)) * w.V * es
    sm = step.slot_map.cpu().numpy()
    moved = int(((sm[..., 0] >= 0) & (sm[..., 0] != sm[..., 1])).sum())
    comp = moved * 2 * 2 * w.H_kv * w.d * es * w.k_cache.shape[0]
    return attention_bytes(w) + ver + comp


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, path=None):
        self.gpu = gpu_index
        self.proc = None
        self.path = path or os.path.join(tempfile.gettempdir(),
                                         f"spec_bench_clocks_{os.getpid()}_{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        sms = sorted(r["sm"] for r in rows)
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


# ---------------------------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on host copies of the workload the GPU ran.
# A unit of work is (request r, a subset of its query heads): tree attention of every tree
# token of r for those heads; the unit that holds r's first head also runs r's tree build,
# verification and KV compaction.  Tree tokens are credited in proportion to the heads covered
# (every (token, head) row of a request costs the same), so the verification's time is counted
# but not credited.
# ---------------------------------------------------------------------------------------------
_ORACLE_DATA = {}


def _oracle_init(shm_name, layout, scalars):
    """Worker initialiser: attach the shared-memory copy of the sampled requests' arrays."""
    import numpy as np
    from multiprocessing import shared_memory
    shm = shared_memory.SharedMemory(name=shm_name)
    _ORACLE_DATA["shm"] = shm
    arrays = {}
    for key, (off, shape, dtype) in layout.items():
        n = int(np.prod(shape)) if shape else 1
        arrays[key] = np.ndarray(shape, dtype=dtype, buffer=shm.buf, offset=off) if n else \
            np.zeros(shape, dtype=dtype)
    _ORACLE_DATA["arrays"] = arrays
    _ORACLE_DATA["scalars"] = scalars


def _oracle_unit(unit):
    """One unit of oracle work (see above); returns its seconds."""
    import numpy as np
    from oracle import attention as OA, compact as OC, tree as OT, verify as OV
    r, heads, full = unit
    a, s = _ORACLE_DATA["arrays"], _ORACLE_DATA["scalars"]
    t0 = time.perf_counter()
    q = a[f"q{r}"]
    par = a[f"par{r}"]
    T = len(par)
    P = int(s["P"][r])
    table = a[f"table{r}"]
    OA.tree_attention(q, a[f"k{r}"], a[f"v{r}"], table, [P], [0, T], par, s["bs"],
                      rows=[(i, h) for h in heads for i in range(T)])
    if full:
        OT.tree_build(par, [0, T], [P], s["T_max"])
        ver = OV.verify(a[f"tgt{r}"], a[f"drf{r}"], s["draft_kind"], a[f"drow{r}"],
                        a[f"tok{r}"], par, [0, T], a[f"uni{r}"], s["tau"], s["V"],
                        s["max_path"], T_max=s["T_max"])
        kc, vc = a[f"k{r}"][None], a[f"v{r}"][None]
        OC.kv_compact(kc.copy(), vc.copy(), table, [P], ver["path"], ver["n_acc"], s["bs"],
                      s["max_path"], status=ver["status"])
    return time.perf_counter() - t0


def oracle_arrays(w, reqs):
    """Host copies (numpy, fp32 where the oracle reads logits / activations) of what the oracle
    needs for requests `reqs`, with each request's draft rows renumbered locally."""
    import numpy as np
    import torch
    no = w.node_offset.cpu().numpy()
    P = w.prefix_len.cpu().numpy()
    out = {}
    for r in reqs:
        o0, o1 = int(no[r]), int(no[r + 1])
        nblk = -(-(int(P[r]) + o1 - o0) // w.bs)
        blocks = w.block_table[r, :nblk].long()
        out[f"k{r}"] = w.k_cache[0].index_select(0, blocks).float().cpu().numpy()
        out[f"v{r}"] = w.v_cache[0].index_select(0, blocks).float().cpu().numpy()
        out[f"table{r}"] = np.arange(nblk, dtype=np.int64)[None, :]
        out[f"q{r}"] = w.q[o0:o1].float().cpu().numpy()
        out[f"par{r}"] = w.parent[o0:o1].cpu().numpy()
        out[f"tok{r}"] = w.tokens[o0:o1].cpu().numpy()
        out[f"uni{r}"] = w.uniforms[o0:o1].cpu().numpy()
        out[f"tgt{r}"] = w.target[o0:o1].float().cpu().numpy()
        drow = w.draft_row[o0:o1].cpu().numpy()
        used = sorted(set(int(x) for x in drow if x >= 0))
        remap = {d: i for i, d in enumerate(used)}
        out[f"drow{r}"] = np.array([remap.get(int(x), -1) for x in drow], dtype=np.int64)
        idx = torch.as_tensor(used if used else [0], dtype=torch.long, device=w.draft.device)
        out[f"drf{r}"] = w.draft.index_select(0, idx).float().cpu().numpy()
    scalars = dict(P=[int(x) for x in P], bs=w.bs, T_max=w.T_max, draft_kind=w.draft_kind,
                   tau=w.tau, V=w.V, max_path=w.max_path)
    return out, scalars


def cpu_baseline(w, budget_s=5.0, cores=None):
    """The oracle timed on the host: a single-core sample and an all-core sample (one spawned
    process per core, the sampled requests' arrays shared through shared memory), each sized to
    about budget_s seconds of wall time.  Returns the cpu_baseline object."""
    import multiprocessing as mp
    import numpy as np
    from concurrent.futures import ProcessPoolExecutor
    from multiprocessing import shared_memory

    cores = cores or len(os.sched_getaffinity(0))
    sizes = w.tree_sizes()
    # probe: one (request 0, one head) unit, in process
    arrs, scalars = oracle_arrays(w, [0])
    _oracle_init_local(arrs, scalars)
    per_head = max(_oracle_unit((0, [0], False)), 1e-4)

    def sample(budget, n_cores):
        # units of about equal cost: (request, head chunk), credited tokens sizes[r] * h / H_q
        target_rows = budget * n_cores / per_head
        units, credited, left, r = [], 0.0, target_rows, 0
        while left > 0 and r < w.B:
            nh = int(min(w.H_q, max(1, round(left))))
            heads = [int(j * w.H_q // nh) for j in range(nh)]
            chunk = max(1, math.ceil(nh / n_cores)) if n_cores > 1 else nh
            for c0 in range(0, nh, chunk):
                units.append((r, heads[c0:c0 + chunk], c0 == 0))
            credited += sizes[r] * nh / w.H_q
            left -= nh
            r += 1
        return units, credited

    res = {"unit": "verified tree tokens/s", "kind": "oracle", "cores": 1}
    # single core
    units1, cred1 = sample(budget_s, 1)
    reqs1 = sorted(set(u[0] for u in units1))
    arrs, scalars = oracle_arrays(w, reqs1)
    _oracle_init_local(arrs, scalars)
    t1 = sum(_oracle_unit(u) for u in units1)
    # a workload smaller than the budget is run again until about half the budget has passed
    reps = max(1, min(1000, int(0.5 * budget_s / max(t1, 1e-6))))
    if reps > 1:
        t1 = sum(_oracle_unit(u) for _ in range(reps) for u in units1)
        units1, cred1 = units1 * reps, cred1 * reps
    res["value"] = cred1 / t1
    res["single_core"] = {"value": cred1 / t1, "cores": 1, "seconds": round(t1, 2),
                          "sample": _sample_text(w, units1, cred1)}
    # all cores
    if cores > 1:
        unitsn, credn = sample(budget_s, cores)
        if reps > 1:   # as many repetitions per core as the single-core leg ran
            unitsn, credn = unitsn * (reps * cores), credn * (reps * cores)
        reqsn = sorted(set(u[0] for u in unitsn))
        arrs, scalars = oracle_arrays(w, reqsn)
        layout, total = {}, 0
        for k, a in arrs.items():
            total = (total + 63) // 64 * 64
            layout[k] = (total, a.shape, a.dtype.str)
            total += a.nbytes
        shm = shared_memory.SharedMemory(create=True, size=max(total, 64))
        try:
            for k, a in arrs.items():
                off, shape, dt = layout[k]
                np.ndarray(shape, dtype=dt, buffer=shm.buf, offset=off)[...] = a
            del arrs
            with ProcessPoolExecutor(cores, mp_context=mp.get_context("spawn"),
                                     initializer=_oracle_init,
                                     initargs=(shm.name, layout, scalars)) as ex:
                list(ex.map(_noop, range(4 * cores)))   # every worker started and attached
                t0 = time.perf_counter()
                list(ex.map(_oracle_unit, unitsn))
                tn = time.perf_counter() - t0
        finally:
            shm.close()
            shm.unlink()
        res["all_cores"] = {"value": credn / tn, "cores": cores, "seconds": round(tn, 2),
                            "sample": _sample_text(w, unitsn, credn)}
        res["value"] = credn / tn
        res["cores"] = cores
    res["sample"] = (f"{res['single_core']['sample']}; all-core: "
                     f"{res.get('all_cores', {}).get('sample', 'n/a')}")
    return res


def _noop(x):
    return x


def _oracle_init_local(arrs, scalars):
    _ORACLE_DATA["arrays"] = arrs
    _ORACLE_DATA["scalars"] = scalars


def _sample_text(w, units, credited):
    reqs = sorted(set(u[0] for u in units))
    heads = sum(len(u[1]) for u in units)
    runs = sum(1 for u in units if u[2])
    return (f"{len(reqs)} of {w.B} requests, {heads} (request, query head) attention units "
            f"({len(reqs) * w.H_q} per pass over them), full vocab and KV, {runs} verification "
            f"+ compaction runs of the sampled requests; {credited:.1f} tree tokens credited "
            f"(tokens x heads covered / {w.H_q}); numpy fp64")


def oracle_parity(w, step):
    """The oracle's verification of the whole batch (fp64, on the GPU run's inputs) against the
    step's outputs: identical requests, exempt divergences (the first difference at a decision
    whose uniform lies within 1e-6 of its boundary), and the number of such near-boundary
    decisions among all decisions the oracle took."""
    import numpy as np
    from oracle import verify as OV
    target = w.target.float().cpu().numpy()
    draft = w.draft.float().cpu().numpy()
    orc = OV.verify(target, draft, w.draft_kind, w.draft_row.cpu().numpy(),
                    w.tokens.cpu().numpy(), w.parent.cpu().numpy(),
                    w.node_offset.cpu().numpy(), w.uniforms.cpu().numpy(), w.tau, w.V,
                    w.max_path, T_max=w.T_max)
    path, toks = step.path.cpu().numpy(), step.out_tokens.cpu().numpy()
    n_acc, out_len, st = step.n_acc.cpu().numpy(), step.out_len.cpu().numpy(), \
        step.req_status.cpu().numpy()

    def near(e):
        return (e[0] == "test" and abs(e[4] - e[3]) < BAND) or (e[0] == "sample" and e[3] < BAND)

    same = exempt = unexplained = 0
    for r in range(w.B):
        if int(st[r]) != int(orc["status"][r]):
            unexplained += 1
            continue
        g_path = path[r, :n_acc[r] + 1].tolist() if n_acc[r] >= 0 else []
        g_tok = toks[r, :out_len[r]].tolist()
        if g_path == orc["path"][r] and g_tok == orc["out_tokens"][r]:
            same += 1
            continue
        k = 0
        while k < min(len(g_path), len(orc["path"][r])) and g_path[k] == orc["path"][r][k]:
            k += 1
        node = orc["path"][r][k - 1] if k > 0 else 0
        if any(near(e) and e[1] == node for e in orc["events"][r]):
            exempt += 1
        else:
            unexplained += 1
    decisions = sum(max(1, len(e)) for e in orc["events"])
    band = sum(1 for es in orc["events"] for e in es if near(e))
    return {"requests": w.B, "identical": same, "exempt_divergences": exempt,
            "unexplained_divergences": unexplained, "decisions": decisions,
            "near_boundary_decisions": band,
            "exempt_fraction_of_decisions": exempt / max(1, decisions)}


def run_oracle_sample(w, n_req):
    """The CPU oracle (as it stands) on the first n_req requests of the workload, every head:
    tree build, attention of every tree token and head, verification and compaction.  Returns
    seconds."""
    arrs, scalars = oracle_arrays(w, list(range(n_req)))
    _oracle_init_local(arrs, scalars)
    return sum(_oracle_unit((r, list(range(w.H_q)), True)) for r in range(n_req))


def rank_seeds(rank):
    """Seeds of rank `rank`'s batch: every rank verifies its own requests of the same shape
    (weak scaling), rank 0 the default workload."""
    return dict(logits=1 + 1000 * rank, drafting=2 + 1000 * rank, qkv=3 + 1000 * rank)


def max_over_ranks(seconds, world, device=None):
    """The slowest rank's time, returned on every rank: the job is done when all ranks are."""
    if world <= 1:
        return seconds
    import torch
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step, steps, seconds, world):
    """Units all ranks processed per second of the slowest rank."""
    return world * units_per_rank_step * steps / seconds


def method_stats(w, step):
    """The method's own numbers for one step: accepted drafts, emitted tokens (accepted drafts
    plus the final token, E[L]) and the acceptance rate (accepted / tested children)."""
    n_acc = step.n_acc.cpu().float()
    rej = step.rejections.cpu().float()
    out_len = step.out_len.cpu().float()
    ok = n_acc >= 0
    acc, tested = float(n_acc[ok].sum()), float((n_acc[ok] + rej[ok]).sum())
    drafts = sum(w.tree_sizes()) - w.B
    return {"accepted_drafts_per_request": round(float(n_acc[ok].mean()), 4),
            "emitted_tokens_per_request": round(float(out_len.mean()), 4),
            "acceptance_rate": round(acc / tested, 4) if tested else None,
            "accepted_over_drafted": round(acc / drafts, 4) if drafts else None,
            "rejected_children_per_request": round(float(rej[ok].mean()), 4)}


# ---------------------------------------------------------------------------------------------
def reference_arm(args, rank):
    """--impl reference: the CPU oracle (fp64, one core) on a bounded sample of the headline
    workload per step; rank 0 alone runs it."""
    if rank != 0:
        return
    from speculative_decoding_draft_tree_gb300 import workloads as W
    w = W.make_config(args.workload, scale="full", device="cpu", batch=args.batch)
    tokens_per_step = int(sum(w.tree_sizes()))
    vals = []
    budget = max(0.5, min(2.0, args.cpu_budget))
    arrs, scalars = oracle_arrays(w, [0])
    _oracle_init_local(arrs, scalars)
    per_head = max(_oracle_unit((0, [0], False)), 1e-4)
    nh_total = max(1, int(budget / per_head))
    units, credited, left, r = [], 0.0, nh_total, 0
    sizes = w.tree_sizes()
    while left > 0 and r < w.B:
        nh = int(min(w.H_q, left))
        units.append((r, [int(j * w.H_q // nh) for j in range(nh)], True))
        credited += sizes[r] * nh / w.H_q
        left -= nh
        r += 1
    arrs, scalars = oracle_arrays(w, sorted(set(u[0] for u in units)))
    _oracle_init_local(arrs, scalars)
    for i in range(args.warmup + args.steps):
        t = sum(_oracle_unit(u) for u in units)
        if i >= args.warmup:
            vals.append(credited / t)
    value = median(vals)
    cb = {"value": value, "unit": "verified tree tokens/s", "cores": 1, "kind": "oracle",
          "sample": _sample_text(w, units, credited)}
    line = {"impl": "reference", "metric": "verified tree tokens/s", "value": value,
            "unit": "verified tree tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * tokens_per_step / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_description(w, args.workload),
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "verified tree tokens/s",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


class Timed:
    """CUDA-event pairs for `steps` timed calls on `stream`."""

    def __init__(self, steps):
        import torch
        self.ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(steps)]

    def ms(self):
        return [a.elapsed_time(b) for a, b in self.ev]


def main():
    args = parse()
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        reference_arm(args, rank)
        return

    import torch
    import torch.distributed as dist
    from speculative_decoding_draft_tree_gb300 import binding
    from speculative_decoding_draft_tree_gb300 import workloads as W
    from speculative_decoding_draft_tree_gb300.api import RoundPipeline, VerifyStep

    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    binding.load_library(build_if_missing=True)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    steps = args.steps
    cids = [args.workload] + [int(c) for c in args.configs.split(",")
                              if c.strip() and int(c) != args.workload]
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def l2_flush(i):
        # the write evicts the step's data; the read of a second buffer then evicts the written
        # (dirty) lines, so the step neither finds its inputs in L2 nor pays for write-backs
        flush_w.fill_(i & 0xFF)
        torch.amax(flush_r)

    # ---- set-up of every workload (weak scaling: every rank verifies its own batch)
    runs = {}
    for cid in cids:
        w = W.make_config(cid, scale="full", device=dev, seeds=rank_seeds(rank),
                          batch=args.batch if cid == args.workload else None)
        step = VerifyStep(w)
        for _ in range(max(3, args.warmup)):
            step.run()
        torch.cuda.synchronize()
        n0 = binding.spec_kernel_launches()
        graph = step.capture_graph()   # the same step as one CUDA graph
        launches = binding.spec_kernel_launches() - n0
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        runs[cid] = dict(w=w, step=step, graph=graph, launches=launches)

    nxt = None if args.no_next else setup_next(args, dev, rank, W, VerifyStep, binding)
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank, args.clocks_csv) if rank == 0 else None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    t_wall0 = time.perf_counter()
    for cid in cids:
        run = runs[cid]
        step, graph = run["step"], run["graph"]
        tg, ts, ta = Timed(steps), Timed(steps), Timed(steps)
        for i in range(steps):   # the headline form: each step replayed as one CUDA graph
            l2_flush(i)
            tg.ev[i][0].record(stream)
            graph.replay()
            tg.ev[i][1].record(stream)
        for i in range(steps):   # the same step launched call by call
            l2_flush(i)
            ts.ev[i][0].record(stream)
            step.run()
            ts.ev[i][1].record(stream)
        for i in range(steps):   # the attention call alone (roofline)
            l2_flush(i)
            step.tree_build()
            ta.ev[i][0].record(stream)
            step.attention()
            ta.ev[i][1].record(stream)
        run.update(tg=tg, ts=ts, ta=ta)
    if nxt is not None:
        time_next(nxt, steps, l2_flush, stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    timed_wall_s = time.perf_counter() - t_wall0

    # end to end through the public API (RoundPipeline) with pinned host buffers: every round's
    # inputs are copied from pinned host memory and its accepted tokens copied back inside the
    # timed region; two steps over separate buffers (same KV cache) let round i + 1's upload
    # overlap round i's kernels, as a serving loop would.  No L2 flush between rounds: each
    # round streams its K/V (4x L2 and more) and the copy engine writes the round's inputs.
    for cid in cids:
        run = runs[cid]
        if args.no_e2e:
            run["e2e"] = None
            continue
        step = run["step"]
        pipe = RoundPipeline(step, stream)
        host_in = pipe.pinned_host_inputs()
        for _ in range(4):
            pipe.submit(host_in)
        pipe.finish()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            pipe.submit(host_in)
        pipe.finish()   # the timed region ends with the last results on the host
        e1.record(stream)
        torch.cuda.synchronize()
        t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
        tokens = int(sum(run["w"].tree_sizes()))
        run["e2e"] = {"value": round(job_throughput(tokens, steps, t_e2e, world), 1),
                      "unit": "verified tree tokens/s",
                      "h2d_bytes_per_step": VerifyStep.bytes_of(host_in),
                      "d2h_bytes_per_step": VerifyStep.bytes_of(pipe.host_outputs(0)),
                      "ms_per_step": round(1e3 * t_e2e / steps, 4)}
        del pipe, host_in

    sweep = None
    if not args.no_sweep:
        sweep = alpha_sweep(dev, rank, W, VerifyStep)

    peaks = measured_peaks()
    results = {}
    for cid in cids:
        run = runs[cid]
        results[cid] = config_result(cid, run, steps, world, dev, peaks, rank, args)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    head = results[args.workload]
    w = runs[args.workload]["w"]
    line = {
        "metric": "verified tree tokens/s", "value": head["value"],
        "unit": "verified tree tokens/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded generators shaped like the pages' workloads)",
        "config": workload_description(w, args.workload),
        "timing": "median of the timed steps, each replayed as one CUDA graph of the step's "
                  "launches, L2 flushed before each; p10 / p90 beside it",
    }
    for k in ("ms_p10", "ms_p90", "requests_per_s", "stream", "step_roofline", "roofline",
              "tensor", "stats", "parity", "cpu_baseline", "e2e", "gpu_launches_per_step"):
        line[k] = head.get(k)
    line["gpu_launches"] = head["gpu_launches_per_step"] * steps
    line["clocks"] = clocks
    line["timed_region_wall_s"] = round(timed_wall_s, 2)
    line["configs"] = {runs[c]["w"].name: results[c] for c in cids if c != args.workload}
    line["alpha_sweep"] = sweep
    line["next"] = None if nxt is None else next_results(nxt, peaks)
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def config_result(cid, run, steps, world, dev, peaks, rank, args):
    """The per-workload object of the JSON line."""
    w, step = run["w"], run["step"]
    tokens = int(sum(w.tree_sizes()))
    g_ms, s_ms, a_ms = run["tg"].ms(), run["ts"].ms(), run["ta"].ms()
    t_step = max_over_ranks(median(g_ms) / 1e3, world, dev)
    t_stream = max_over_ranks(median(s_ms) / 1e3, world, dev)
    t_attn = median(a_ms) / 1e3
    abytes = attention_bytes(w)
    sbytes = step_bytes(w, step)
    aflops = attention_flops(w)
    achieved = abytes / t_attn / 1e9
    res = {
        "workload": w.name, "tree_tokens_per_step": tokens, "batch_requests": w.B,
        "value": round(job_throughput(tokens, 1, t_step, world), 1),
        "unit": "verified tree tokens/s",
        "ms_per_step": round(1e3 * t_step, 4),
        "ms_p10": round(percentile(g_ms, 10), 4), "ms_p90": round(percentile(g_ms, 90), 4),
        "requests_per_s": round(world * w.B / t_step, 1),
        "stream": {"ms_per_step": round(1e3 * t_stream, 4),
                   "value": round(job_throughput(tokens, 1, t_stream, world), 1)},
        "step_roofline": {"bound": "hbm", "algorithmic_bytes": sbytes,
                          "achieved": round(sbytes / t_step / 1e9, 1), "peak": peaks["hbm"],
                          "unit": "GB/s", "frac": round(sbytes / t_step / 1e9 / peaks["hbm"], 4),
                          "frac_of_nominal": round(sbytes / t_step / 1e9 / NOMINAL_HBM_GBS, 4),
                          "peak_kind": peaks["kind"]},
        "roofline": {"bound": "hbm", "kernel": "spec_tree_attention (tcgen05 main + merge)"
                     if w.dtype == "bf16" else "spec_tree_attention (fp32 CUDA-core kernel)",
                     "achieved": round(achieved, 1), "peak": peaks["hbm"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm"], 4),
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "traffic": recorded_traffic(w.name), "peak_kind": peaks["kind"],
                     "algorithmic_bytes": abytes, "us_per_launch": round(t_attn * 1e6, 2),
                     "us_p10": round(percentile(a_ms, 10) * 1e3, 2),
                     "us_p90": round(percentile(a_ms, 90) * 1e3, 2)},
        "tensor": {"flops_per_launch": aflops,
                   "achieved_tflops": round(aflops / t_attn / 1e12, 1),
                   "peak_tflops": peaks["bf16"],
                   "frac": round(aflops / t_attn / 1e12 / peaks["bf16"], 4),
                   "note": "useful QK^T + PV flops of the visible keys; the kernel also "
                           "multiplies padding rows of partly filled 128-row tiles"},
        "gpu_launches_per_step": run["launches"],
        "stats": method_stats(w, step),
        "e2e": run.get("e2e"),
        "parity": None, "cpu_baseline": None,
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["parity"] = oracle_parity(w, step)
        res["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    return res


def alpha_sweep(dev, rank, W, VerifyStep):
    """Acceptance on the Leviathan chain shape (16 chains of gamma = 5, vocab 32000) for draft
    noise sigma in {0.5, 1, 2} and tau in {0, 1}, over 8 batches of fresh draws (128 chains per
    cell): the measured acceptance rate a (accepted / tested drafts), the emitted tokens per
    request E[L], the closed form (1 - a^(g+1)) / (1 - a) at the measured a, and the mean
    sum_x min(p, q) (tau = 1) or argmax agreement (tau = 0) of the rows, i.e. the acceptance
    probability of a fresh draft from each row."""
    import torch
    out = []
    gamma = 5
    for tau in (1.0, 0.0):
        for sigma in (0.5, 1.0, 2.0):
            acc = tested = 0.0
            lens, a_rows = [], []
            for rep in range(8):
                seeds = dict(logits=101 + 17 * rep + 1000 * rank, drafting=202 + 17 * rep,
                             qkv=3, uniform=rep + 1)
                w = W.chain_workload(B=16, gamma=gamma, V=32000, dtype="bf16", H_q=4, H_kv=4,
                                     d=128, prefix=16, tau=tau, target_std=3.0,
                                     noise_std=sigma, device=dev, contiguous=True,
                                     seeds=seeds)
                step = VerifyStep(w)
                step.tree_build()
                step.verify()
                n_acc = step.n_acc.float()
                acc += float(n_acc.sum())
                tested += float((n_acc + step.rejections.float()).sum())
                lens.append(step.out_len.float())
                internal = w.draft_row >= 0
                tgt = w.target[internal][:, :w.V].float()
                drf = w.draft[w.draft_row[internal].long()][:, :w.V].float()
                if tau > 0:
                    p = torch.softmax(tgt / tau, -1)
                    q = torch.softmax(drf / tau, -1)
                    a_rows.append(torch.minimum(p, q).sum(-1))
                else:
                    a_rows.append((tgt.argmax(-1) == drf.argmax(-1)).float())
            a = acc / tested if tested else float("nan")
            el = float(torch.cat(lens).mean())
            a_exact = float(torch.cat(a_rows).mean())
            closed = (1 - a ** (gamma + 1)) / (1 - a) if a < 1 else gamma + 1.0
            closed_exact = (1 - a_exact ** (gamma + 1)) / (1 - a_exact) if a_exact < 1 \
                else gamma + 1.0
            out.append({"sigma": sigma, "tau": tau, "chains": 128,
                        "acceptance_rate": round(a, 4), "emitted_tokens_per_request": round(el, 4),
                        "closed_form_at_measured_rate": round(closed, 4),
                        "row_acceptance_probability": round(a_exact, 4),
                        "closed_form_at_row_probability": round(closed_exact, 4)})
    return out


# ---------------------------------------------------------------------------------------------
# Rows after the path: measured beside the step.
# ---------------------------------------------------------------------------------------------
def setup_next(args, dev, rank, W, VerifyStep, binding):
    import torch
    from speculative_decoding_draft_tree_gb300.api import DraftTreeBuilder
    n = {}
    # the step before attention (rotary embedding + tree K/V slot write) on the chain workload
    w2 = W.make_config(2, scale="full", device=dev, seeds=rank_seeds(rank))
    step_r = VerifyStep(w2)
    k_new, v_new = W.new_tree_kv(w2)
    step_r.enable_rope(w2.q.clone(), k_new, v_new)
    step_p = VerifyStep(w2)
    for _ in range(3):
        step_r.run()
        step_p.run()
    n.update(w2=w2, step_r=step_r, step_p=step_p)
    # the lookahead-decoding forward (2-D Jacobi window + candidate n-grams)
    wl = W.lookahead_config(scale="full", device=dev, seeds=rank_seeds(rank))
    step_l = VerifyStep(wl)
    for _ in range(3):
        step_l.run()
    n.update(wl=wl, step_l=step_l)
    # multi-draft verification (5 draft models' chains, every sibling with its own q)
    wm = W.multidraft_config(scale="full", device=dev, seeds=rank_seeds(rank))
    step_m = VerifyStep(wm, sibling_rule=binding.SPEC_SIBLING_MULTI_DRAFT)
    for _ in range(3):
        step_m.run()
    n.update(wm=wm, step_m=step_m)
    # building the draft tree on the device (EAGLE-2 top-5 expansion to depth 8, ECHO budget
    # 2048) on the EAGLE-2 workload's shape; the draft model's rows of all levels resident
    DT_B, DT_K, DT_D, DT_V, DT_KMAX = 64, 5, 8, 152064, 2048
    dt_scales = [0.3 + 3.7 * ((17 * r) % 64) / 63.0 for r in range(DT_B)]
    dt_rows = [W.draft_level_rows(B=DT_B, K=DT_K, V=DT_V, level=lv, device=dev,
                                  seed=11 + rank, scales=dt_scales) for lv in range(1, DT_D + 1)]
    dt_roots = torch.arange(DT_B, dtype=torch.int32, device=dev) * 37 % DT_V
    builder = DraftTreeBuilder(DT_B, DT_K, DT_D, dev)
    n.update(dt=dict(B=DT_B, K=DT_K, D=DT_D, V=DT_V, KMAX=DT_KMAX, rows=dt_rows,
                     roots=dt_roots, builder=builder))
    for _ in range(3):
        build_tree(n["dt"])
    return n


def build_tree(dt):
    b = dt["builder"]
    b.init(dt["roots"])
    for lv in range(1, dt["D"] + 1):
        b.expand(lv)
        b.append(lv, dt["rows"][lv - 1], dt["V"])
    b.echo(dt["KMAX"])


def time_next(n, steps, l2_flush, stream):
    T = {k: Timed(steps) for k in ("rope", "fused", "tree", "step_r", "step_p", "look_attn",
                                   "look_step", "dt", "dt_append", "dt_echo", "multi_ver",
                                   "multi_step")}
    n["T"] = T

    def timed(key, i, fn, before=None):
        l2_flush(i)
        if before:
            before()
        T[key].ev[i][0].record(stream)
        fn()
        T[key].ev[i][1].record(stream)

    step_r, step_p, step_l, step_m = n["step_r"], n["step_p"], n["step_l"], n["step_m"]
    dt = n["dt"]
    b = dt["builder"]
    for i in range(steps):
        timed("rope", i, step_r.rope, before=step_r.tree_build)
        timed("tree", i, step_r.tree_build)
        timed("fused", i, step_r.tree_build_rope)
        timed("step_r", i, step_r.run)
        timed("step_p", i, step_p.run)
        timed("look_attn", i, step_l.attention, before=step_l.tree_build)
        timed("look_step", i, step_l.run)
        timed("dt", i, lambda: build_tree(dt))

        def to_level2():
            b.init(dt["roots"])
            for lv in (1, 2):
                b.expand(lv)
                if lv == 1:
                    b.append(lv, dt["rows"][0], dt["V"])

        timed("dt_append", i, lambda: b.append(2, dt["rows"][1], dt["V"]), before=to_level2)

        def to_echo():
            for lv in range(3, dt["D"] + 1):
                b.expand(lv)
                b.append(lv, dt["rows"][lv - 1], dt["V"])

        timed("dt_echo", i, lambda: b.echo(dt["KMAX"]), before=to_echo)

        def to_verify():
            step_m.tree_build()
            step_m.attention()

        timed("multi_ver", i, step_m.verify, before=to_verify)
        timed("multi_step", i, step_m.run)


def next_results(n, peaks):
    T = n["T"]

    def med_s(key):
        return median(T[key].ms()) / 1e3

    w2, wl, wm, dt = n["w2"], n["wl"], n["wm"], n["dt"]
    tokens2 = int(sum(w2.tree_sizes()))
    rbytes = rope_bytes(w2)
    t_fused, t_step_r, t_step_p = med_s("fused"), med_s("step_r"), med_s("step_p")
    out = {"rope_kv_write": {
        "workload": w2.name,
        "kernel": "spec_tree_build_rope_kv_write (tree build fused with the rotary step)",
        "bound": "hbm", "algorithmic_bytes": rbytes,
        "us_per_launch": round(t_fused * 1e6, 2),
        "achieved": round(rbytes / t_fused / 1e9, 1), "peak": peaks["hbm"], "unit": "GB/s",
        "frac": round(rbytes / t_fused / 1e9 / peaks["hbm"], 4),
        "us_tree_build_alone": round(med_s("tree") * 1e6, 2),
        "us_standalone_rope_call": round(med_s("rope") * 1e6, 2),
        "ms_per_step_with_it": round(1e3 * t_step_r, 4),
        "ms_per_step_plain": round(1e3 * t_step_p, 4),
        "value_with_it": round(tokens2 / t_step_r, 1),
        "timing": "both steps launched call by call, L2 flushed before each"}}
    lbytes = attention_bytes(wl)
    t_la, t_ls = med_s("look_attn"), med_s("look_step")
    look_tokens = int(sum(wl.tree_sizes()))
    out["lookahead"] = {
        "workload": wl.name, "tree_tokens_per_step": look_tokens,
        "kernel": "spec_tree_attention on the lookahead mask", "bound": "hbm",
        "algorithmic_bytes": lbytes, "us_per_launch": round(t_la * 1e6, 2),
        "achieved": round(lbytes / t_la / 1e9, 1), "peak": peaks["hbm"], "unit": "GB/s",
        "frac": round(lbytes / t_la / 1e9 / peaks["hbm"], 4),
        "traffic": recorded_traffic(wl.name),
        "ms_per_step": round(1e3 * t_ls, 4), "value": round(look_tokens / t_ls, 1)}
    # level 2 expands the 5 children of every root: 64 x 5 rows of 152064 bf16 logits
    dt_bytes = dt["B"] * dt["K"] * dt["V"] * 2
    t_app = med_s("dt_append")
    out["draft_tree"] = {
        "workload": f"eagle2 top-{dt['K']} expansion, depth {dt['D']}, {dt['B']} requests, "
                    f"vocab {dt['V']}, ECHO K_max {dt['KMAX']}",
        "kernel": "spec_draft_topk_append (one expansion level, 320 rows)", "bound": "hbm",
        "algorithmic_bytes": dt_bytes, "us_per_launch": round(t_app * 1e6, 2),
        "achieved": round(dt_bytes / t_app / 1e9, 1), "peak": peaks["hbm"], "unit": "GB/s",
        "frac": round(dt_bytes / t_app / 1e9 / peaks["hbm"], 4),
        "us_whole_construction": round(med_s("dt") * 1e6, 2),
        "us_echo_select_pack": round(med_s("dt_echo") * 1e6, 2),
        "tree_tokens": int(dt["builder"].node_offset[-1])}
    multi_tokens = int(sum(wm.tree_sizes()))
    step_m = n["step_m"]
    t_ms = med_s("multi_step")
    out["multidraft"] = {
        "workload": wm.name, "tree_tokens_per_step": multi_tokens,
        "kernel": "spec_verify, multi-draft sibling rule (rows + walk kernels)",
        "bound": "latency", "us_verify_call": round(med_s("multi_ver") * 1e6, 2),
        "rejections_per_request": round(float(step_m.rejections.float().mean()), 3),
        "accepted_tokens_per_request": round(float(step_m.out_len.float().mean()), 3),
        "ms_per_step": round(1e3 * t_ms, 4), "value": round(multi_tokens / t_ms, 1)}
    return out


if __name__ == "__main__":
    main()
