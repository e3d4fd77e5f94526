"""Benchmark of one draft-tree verification round on GB300.

A step = one pass of the whole hot path over one batch of synthetic requests:
spec_tree_build + spec_tree_attention (one layer) + spec_verify_compact (verification and KV
compaction), all through the C-ABI library.  Default workload: the Leviathan chain (16 requests x (1 root + 5 drafts),
vocab 32000, 32 x d128 MHA heads, 2048 cached tokens per request, bf16, tau = 1).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload CID] [--impl reference]

Prints ONE JSON line (rank 0).  `value` is verified tree tokens per second over all ranks
(device time of the K timed steps, each replayed as one CUDA graph of the step's launches,
max over ranks; `stream` gives the same step launched call by call); `step_roofline` divides
the whole step's algorithmic bytes by that time; `e2e` repeats the measurement through the
public RoundPipeline (VerifyStep.upload / run / download) with every round's inputs copied from
pinned host memory and its accepted tokens copied back inside the timed region (two steps
alternate so that the next round's upload overlaps the current round).  `roofline` is for the tree-attention
call (the dominant kernel), with algorithmic bytes = the KV of every request read once + Q + O +
LSE.  `next` measures the step before attention (rotary embedding at the tree's position ids
plus the tree K/V slot write) alone and inside a step that includes it, and the lookahead-
decoding forward (a second mask workload on the same kernels), multi-draft verification and
the device-side construction of the draft tree (EAGLE-2 expansion + ECHO budget).
`--impl reference` times the CPU oracle on a bounded sample of the same workload instead.
"""
import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = 2
# kernels of the library launched by one step of the default workload: tree_build_kernel,
# attn_tc_small_kernel, attn_merge_kernel, verify_cluster_kernel (the one-launch verification
# that trees of up to 32 nodes take, with the KV compaction in the same launch)
KERNELS_PER_STEP = 4
FLUSH_BYTES = 256 << 20
NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e, nominal (the measured copy bandwidth is `peak`)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-requests", type=int, default=0)
    ap.add_argument("--clocks-csv", default=None,
                    help="keep the nvidia-smi samples taken during the timed region in this file")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def workload_description(w, cid):
    from speculative_decoding_draft_tree_gb300 import workloads as W
    sizes = w.tree_sizes()
    P = w.prefix_len.cpu().tolist()
    return {
        "workload": W.CONFIG_NAMES[cid],
        "batch_requests": w.B,
        "tree_tokens_per_step": int(sum(sizes)),
        "drafts_per_step": int(sum(sizes) - w.B),
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


def recorded_traffic():
    """DRAM bytes per launch of the attention kernel from the committed ncu capture, or None
    when the kernel sources changed since the capture was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "attention_traffic.json")
    try:
        rec = json.load(open(path))
        h = hashlib.sha256()
        for src in rec["sources"]:
            h.update(open(os.path.join(ROOT, src), "rb").read())
        if h.hexdigest() != rec["sources_sha256"]:
            return None
        return rec["dram_bytes_read_per_launch"] + rec["dram_bytes_write_per_launch"]
    except Exception:
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
def run_oracle_sample(w, n_req):
    """The CPU oracle (as it stands) on the first n_req requests of the workload: tree build,
    attention of every tree token and head, verification and compaction.  Returns seconds."""
    import numpy as np
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from oracle import attention as OA, compact as OC, tree as OT, verify as OV
    no = w.node_offset.cpu().numpy()
    P = w.prefix_len.cpu().numpy()
    o_end = int(no[n_req])
    parent = w.parent.cpu().numpy()[:o_end]
    nodeoff = no[:n_req + 1]
    q = w.q[:o_end].float().cpu().numpy()
    nblk_need = [-(-(int(P[r]) + int(no[r + 1] - no[r])) // w.bs) for r in range(n_req)]
    table_full = w.block_table.cpu().numpy()[:n_req]
    used = sorted(set(int(b) for r in range(n_req) for b in table_full[r, :nblk_need[r]]))
    remap = {b: i for i, b in enumerate(used)}
    table = np.full_like(table_full, -1)
    for r in range(n_req):
        for j in range(nblk_need[r]):
            table[r, j] = remap[int(table_full[r, j])]
    import torch
    idx = torch.as_tensor(used, dtype=torch.long, device=w.k_cache.device)
    kc = w.k_cache[:, idx].float().cpu().numpy()
    vc = w.v_cache[:, idx].float().cpu().numpy()
    target = w.target[:o_end].float().cpu().numpy()
    draft = w.draft.float().cpu().numpy()
    draft_row = w.draft_row.cpu().numpy()[:o_end]
    tokens = w.tokens.cpu().numpy()[:o_end]
    uni = w.uniforms.cpu().numpy()[:o_end]
    t0 = time.perf_counter()
    tb = OT.tree_build(parent, nodeoff, P[:n_req], w.T_max)
    OA.tree_attention(q, kc[0], vc[0], table, P[:n_req], nodeoff, parent, w.bs)
    ver = OV.verify(target, draft, w.draft_kind, draft_row, tokens, parent, nodeoff, uni, w.tau,
                    w.V, w.max_path, T_max=w.T_max)
    OC.kv_compact(kc, vc, table, P[:n_req], ver["path"], ver["n_acc"], w.bs, w.max_path,
                  status=ver["status"])
    del tb
    return time.perf_counter() - t0


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


def cpu_baseline(w, n_req=None, budget_s=15.0):
    """Time the oracle on a bounded sample sized to about `budget_s` seconds."""
    sizes = w.tree_sizes()
    if n_req is None or n_req <= 0:
        probe = run_oracle_sample(w, 1)
        n_req = max(1, min(w.B, int(budget_s / max(probe, 1e-3))))
    secs = run_oracle_sample(w, n_req)
    tokens = sum(sizes[:n_req])
    return {"value": tokens / secs, "unit": "verified tree tokens/s", "cores": 1,
            "kind": "oracle",
            "sample": f"{n_req} of {w.B} requests ({tokens} tree tokens), full vocab and KV, "
                      f"{secs:.1f} s single-threaded numpy fp64"}


# ---------------------------------------------------------------------------------------------
def main():
    args = parse()
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    rank, world, local_rank = dist_env()
    import torch
    from speculative_decoding_draft_tree_gb300 import workloads as W

    if args.impl == "reference":
        if rank != 0:
            return
        w = W.make_config(args.workload, scale="full", device="cpu")
        tokens_per_step = int(sum(w.tree_sizes()))
        steps = []
        n_req = args.cpu_sample_requests or None
        for i in range(args.warmup + args.steps):
            cb = cpu_baseline(w, n_req=n_req, budget_s=4.0)
            n_req = int(cb["sample"].split(" of ")[0])
            if i >= args.warmup:
                steps.append(cb["value"])
        value = sum(steps) / len(steps)
        cb["value"] = value
        line = {"impl": "reference", "metric": "verified tree tokens/s", "value": value,
                "unit": "verified tree tokens/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": 1e3 * tokens_per_step / value,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": workload_description(w, args.workload),
                "cpu_baseline": cb,
                "e2e": {"value": value, "unit": "verified tree tokens/s",
                        "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch.distributed as dist
    from speculative_decoding_draft_tree_gb300 import binding
    from speculative_decoding_draft_tree_gb300.api import VerifyStep

    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    binding.load_library(build_if_missing=True)
    dev = torch.device("cuda", local_rank)
    # weak scaling: every rank verifies its own batch of the same shape
    w = W.make_config(args.workload, scale="full", device=dev, seeds=rank_seeds(rank))
    tokens_per_step = int(sum(w.tree_sizes()))
    step = VerifyStep(w)
    stream = torch.cuda.current_stream()
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def l2_flush(i):
        # the write evicts the step's data; the read of a second buffer then evicts the written
        # (dirty) lines, so the step neither finds its inputs in L2 nor pays for write-backs
        flush_w.fill_(i & 0xFF)
        torch.amax(flush_r)

    for _ in range(max(3, args.warmup)):
        step.run()
    torch.cuda.synchronize()
    # the same step as one CUDA graph (the launches keep their programmatic dependencies)
    step_graph = step.capture_graph()
    for _ in range(3):
        step_graph.replay()
    torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    ev_attn = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    # the step before attention (rotary embedding + tree K/V slot write), measured beside the
    # step: alone, and as part of a step that includes it
    step_r = VerifyStep(w)
    k_new, v_new = W.new_tree_kv(w)
    step_r.enable_rope(w.q.clone(), k_new, v_new)
    def ev_pairs():
        return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]

    ev_rope, ev_fused, ev_tree, ev_step_r = ev_pairs(), ev_pairs(), ev_pairs(), ev_pairs()
    ev_graph = ev_pairs()
    for _ in range(3):
        step_r.run()
    # the lookahead-decoding forward (2-D Jacobi window + candidate n-grams) as a second mask
    # workload on the same kernels: its attention call alone and a whole greedy step
    wl = W.lookahead_config(scale="full", device=dev, seeds=rank_seeds(rank))
    step_l = VerifyStep(wl)
    ev_look_attn, ev_look_step = ev_pairs(), ev_pairs()
    for _ in range(3):
        step_l.run()
    # multi-draft verification (5 draft models' chains, every sibling with its own q)
    wm = W.multidraft_config(scale="full", device=dev, seeds=rank_seeds(rank))
    step_m = VerifyStep(wm, sibling_rule=binding.SPEC_SIBLING_MULTI_DRAFT)
    ev_multi_ver, ev_multi_step = ev_pairs(), ev_pairs()
    for _ in range(3):
        step_m.run()
    # building the draft tree on the device (EAGLE-2 top-5 expansion to depth 8, ECHO budget
    # 2048) on the EAGLE-2 workload's shape; the draft model's rows of all levels resident
    from speculative_decoding_draft_tree_gb300.api import DraftTreeBuilder
    DT_B, DT_K, DT_D, DT_V, DT_KMAX = 64, 5, 8, 152064, 2048
    dt_scales = [0.3 + 3.7 * ((17 * r) % 64) / 63.0 for r in range(DT_B)]
    dt_rows = [W.draft_level_rows(B=DT_B, K=DT_K, V=DT_V, level=lv, device=dev,
                                  seed=11 + rank, scales=dt_scales) for lv in range(1, DT_D + 1)]
    dt_roots = torch.arange(DT_B, dtype=torch.int32, device=dev) * 37 % DT_V
    builder = DraftTreeBuilder(DT_B, DT_K, DT_D, dev)

    def build_tree():
        builder.init(dt_roots)
        for lv in range(1, DT_D + 1):
            builder.expand(lv)
            builder.append(lv, dt_rows[lv - 1], DT_V)
        builder.echo(DT_KMAX)

    ev_dt, ev_dt_append, ev_dt_echo = ev_pairs(), ev_pairs(), ev_pairs()
    for _ in range(3):
        build_tree()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank, args.clocks_csv) if rank == 0 else None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    # whole steps: only the step boundaries are recorded, so nothing breaks the overlap of
    # consecutive launches inside a step
    for i in range(args.steps):
        l2_flush(i)
        s0, s1 = ev[i]
        s0.record(stream)
        step.run()
        s1.record(stream)
    # the same step replayed as one CUDA graph, same flush
    for i in range(args.steps):
        l2_flush(i)
        g0, g1 = ev_graph[i]
        g0.record(stream)
        step_graph.replay()
        g1.record(stream)
    # the attention call alone (roofline), same flush, on the same stream
    for i in range(args.steps):
        l2_flush(i)
        step.tree_build()
        a0, a1 = ev_attn[i]
        a0.record(stream)
        step.attention()
        a1.record(stream)
    for i in range(args.steps):   # the standalone rotary call, after a tree build
        l2_flush(i)
        step_r.tree_build()
        r0, r1 = ev_rope[i]
        r0.record(stream)
        step_r.rope()
        r1.record(stream)
    for i in range(args.steps):   # the tree build alone, and fused with the rotary step
        l2_flush(i)
        r0, r1 = ev_tree[i]
        r0.record(stream)
        step_r.tree_build()
        r1.record(stream)
        l2_flush(i)
        r0, r1 = ev_fused[i]
        r0.record(stream)
        step_r.tree_build_rope()
        r1.record(stream)
    for i in range(args.steps):   # a whole step with the fused launch
        l2_flush(i)
        r0, r1 = ev_step_r[i]
        r0.record(stream)
        step_r.run()
        r1.record(stream)
    for i in range(args.steps):   # the lookahead forward: attention alone, then a whole step
        l2_flush(i)
        step_l.tree_build()
        r0, r1 = ev_look_attn[i]
        r0.record(stream)
        step_l.attention()
        r1.record(stream)
        l2_flush(i)
        r0, r1 = ev_look_step[i]
        r0.record(stream)
        step_l.run()
        r1.record(stream)
    for i in range(args.steps):   # draft tree: the whole construction; one full level's top-K
        l2_flush(i)
        r0, r1 = ev_dt[i]
        r0.record(stream)
        build_tree()
        r1.record(stream)
        builder.init(dt_roots)
        for lv in (1, 2):
            builder.expand(lv)
            if lv == 1:
                builder.append(lv, dt_rows[0], DT_V)
        l2_flush(i)
        r0, r1 = ev_dt_append[i]
        r0.record(stream)
        builder.append(2, dt_rows[1], DT_V)
        r1.record(stream)
        for lv in range(3, DT_D + 1):
            builder.expand(lv)
            builder.append(lv, dt_rows[lv - 1], DT_V)
        l2_flush(i)
        r0, r1 = ev_dt_echo[i]
        r0.record(stream)
        builder.echo(DT_KMAX)
        r1.record(stream)
    for i in range(args.steps):   # multi-draft: the verify call alone, then a whole step
        l2_flush(i)
        step_m.tree_build()
        step_m.attention()
        r0, r1 = ev_multi_ver[i]
        r0.record(stream)
        step_m.verify()
        r1.record(stream)
        l2_flush(i)
        r0, r1 = ev_multi_step[i]
        r0.record(stream)
        step_m.run()
        r1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    attn_ms = [e[0].elapsed_time(e[1]) for e in ev_attn]
    def mean_s(evs):
        return sum(e[0].elapsed_time(e[1]) for e in evs) / len(evs) / 1e3

    t_rope, t_fused, t_tree, t_step_r = (mean_s(ev_rope), mean_s(ev_fused), mean_s(ev_tree),
                                         mean_s(ev_step_r))
    t_look_attn, t_look_step = mean_s(ev_look_attn), mean_s(ev_look_step)
    t_graph = max_over_ranks(mean_s(ev_graph), world, dev)
    t_multi_ver, t_multi_step = mean_s(ev_multi_ver), mean_s(ev_multi_step)
    t_dt, t_dt_append, t_dt_echo = mean_s(ev_dt), mean_s(ev_dt_append), mean_s(ev_dt_echo)
    t_stream = max_over_ranks(sum(step_ms) / 1e3, world, dev)
    t_attn = sum(attn_ms) / len(attn_ms) / 1e3
    # the headline: the step timed as one CUDA graph (its launches keep their programmatic
    # dependencies), K replays with the L2 flushed before each; the same step launched call by
    # call is reported beside it ("stream")
    t_total = t_graph * args.steps
    ms_per_step = 1e3 * t_graph
    value = job_throughput(tokens_per_step, args.steps, t_total, world)

    # end to end through the public API (RoundPipeline) with pinned host buffers: every round's
    # inputs are copied from pinned host memory and its accepted tokens copied back inside the
    # timed region; two steps over separate buffers (same KV cache) let round i + 1's upload
    # overlap round i's kernels, as a serving loop would.  No L2 flush between rounds:
    # each round streams 540 MB of K/V (4x L2) and the copy engine writes the round's inputs.
    e2e = None
    if not args.no_e2e:
        from speculative_decoding_draft_tree_gb300.api import RoundPipeline
        pipe = RoundPipeline(step, stream)
        host_in = pipe.pinned_host_inputs()
        for _ in range(4):
            pipe.submit(host_in)
        pipe.finish()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            pipe.submit(host_in)
        pipe.finish()   # the timed region ends with the last results on the host
        e1.record(stream)
        torch.cuda.synchronize()
        t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
        e2e = {"value": job_throughput(tokens_per_step, args.steps, t_e2e, world),
               "unit": "verified tree tokens/s",
               "h2d_bytes_per_step": VerifyStep.bytes_of(host_in),
               "d2h_bytes_per_step": VerifyStep.bytes_of(pipe.host_outputs(0)),
               "ms_per_step": 1e3 * t_e2e / args.steps}

    if rank != 0:
        dist.destroy_process_group() if world > 1 else None
        return
    peak, peak_kind = measured_peaks()
    abytes = attention_bytes(w)
    sbytes = step_bytes(w, step)
    achieved = abytes / t_attn / 1e9
    out_len = step.out_len.cpu()
    roofline = {"bound": "hbm", "kernel": "spec_tree_attention (tcgen05 main + merge)",
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                "traffic": recorded_traffic() if args.workload == DEFAULT_WORKLOAD else None,
                "peak_kind": peak_kind, "algorithmic_bytes": abytes,
                "us_per_launch": round(t_attn * 1e6, 2)}
    rbytes = rope_bytes(w)
    next_rows = {"rope_kv_write": {
        "kernel": "spec_tree_build_rope_kv_write (tree build fused with the rotary step)",
        "bound": "hbm", "algorithmic_bytes": rbytes,
        "us_per_launch": round(t_fused * 1e6, 2),
        "achieved": round(rbytes / t_fused / 1e9, 1), "peak": peak, "unit": "GB/s",
        "frac": round(rbytes / t_fused / 1e9 / peak, 4),
        "us_tree_build_alone": round(t_tree * 1e6, 2),
        "us_standalone_rope_call": round(t_rope * 1e6, 2),
        "ms_per_step_with_it": round(1e3 * t_step_r, 4),
        "value_with_it": round(tokens_per_step / t_step_r, 1)}}
    lbytes = attention_bytes(wl)
    look_tokens = int(sum(wl.tree_sizes()))
    next_rows["lookahead"] = {
        "workload": wl.name, "tree_tokens_per_step": look_tokens,
        "kernel": "spec_tree_attention on the lookahead mask", "bound": "hbm",
        "algorithmic_bytes": lbytes, "us_per_launch": round(t_look_attn * 1e6, 2),
        "achieved": round(lbytes / t_look_attn / 1e9, 1), "peak": peak, "unit": "GB/s",
        "frac": round(lbytes / t_look_attn / 1e9 / peak, 4),
        "ms_per_step": round(1e3 * t_look_step, 4),
        "value": round(look_tokens / t_look_step, 1)}
    # level 2 expands the 5 children of every root: 64 x 5 rows of 152064 bf16 logits
    dt_bytes = DT_B * DT_K * DT_V * 2
    next_rows["draft_tree"] = {
        "workload": f"eagle2 top-{DT_K} expansion, depth {DT_D}, {DT_B} requests, vocab {DT_V},"
                    f" ECHO K_max {DT_KMAX}",
        "kernel": "spec_draft_topk_append (one expansion level, 320 rows)", "bound": "hbm",
        "algorithmic_bytes": dt_bytes, "us_per_launch": round(t_dt_append * 1e6, 2),
        "achieved": round(dt_bytes / t_dt_append / 1e9, 1), "peak": peak, "unit": "GB/s",
        "frac": round(dt_bytes / t_dt_append / 1e9 / peak, 4),
        "us_whole_construction": round(t_dt * 1e6, 2),
        "us_echo_select_pack": round(t_dt_echo * 1e6, 2),
        "tree_tokens": int(builder.node_offset[-1])}
    multi_tokens = int(sum(wm.tree_sizes()))
    next_rows["multidraft"] = {
        "workload": wm.name, "tree_tokens_per_step": multi_tokens,
        "kernel": "spec_verify, multi-draft sibling rule (rows + walk kernels)",
        "bound": "latency", "us_verify_call": round(t_multi_ver * 1e6, 2),
        "rejections_per_request": round(float(step_m.rejections.float().mean()), 3),
        "accepted_tokens_per_request": round(float(step_m.out_len.float().mean()), 3),
        "ms_per_step": round(1e3 * t_multi_step, 4),
        "value": round(multi_tokens / t_multi_step, 1)}
    cb = None
    if not args.no_cpu_baseline:
        w_cpu = W.make_config(args.workload, scale="full", device="cpu")
        cb = cpu_baseline(w_cpu, n_req=args.cpu_sample_requests or None)
    line = {
        "metric": "verified tree tokens/s", "value": round(value, 1),
        "unit": "verified tree tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic", "config": workload_description(w, args.workload),
        "requests_per_s": round(world * w.B * args.steps / t_total, 1),
        "timing": "each step replayed as one CUDA graph, L2 flushed before each (the stream "
                  "object: the same step launched call by call)",
        "stream": {"ms_per_step": round(1e3 * t_stream / args.steps, 4),
                   "value": round(job_throughput(tokens_per_step, args.steps, t_stream, world), 1)},
        "step_roofline": {"bound": "hbm", "algorithmic_bytes": sbytes,
                          "achieved": round(sbytes / t_graph / 1e9, 1), "peak": peak,
                          "unit": "GB/s", "frac": round(sbytes / t_graph / 1e9 / peak, 4),
                          "frac_of_nominal": round(sbytes / t_graph / 1e9 / NOMINAL_HBM_GBS, 4)},
        "accepted_tokens_per_request": round(float(out_len.float().mean()), 3),
        "roofline": roofline, "cpu_baseline": cb, "e2e": e2e, "next": next_rows,
        "clocks": clocks, "gpu_launches": KERNELS_PER_STEP * args.steps,
    }
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
