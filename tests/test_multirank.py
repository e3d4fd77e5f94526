"""The N > 1 path on CPU: two gloo ranks, as the benchmark runs one rank per GPU.  Every rank
verifies its own batch (no collective on the data path); the only cross-rank step is the max of
the elapsed times.  Also the reference arm under torch.distributed.run: rank 0 alone prints."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_two_gloo_ranks():
    port = _free_port()
    env = dict(os.environ, OMP_NUM_THREADS="1")
    procs = [subprocess.Popen([sys.executable, os.path.join(ROOT, "tests", "multirank_rank.py"),
                               str(r), "2", str(port)], cwd=ROOT, env=env,
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(2)]
    res = []
    for p in procs:
        out, err = p.communicate(timeout=300)
        assert p.returncode == 0, err[-2000:]
        res.append(json.loads([l for l in out.splitlines() if l.startswith("{")][-1]))
    res.sort(key=lambda d: d["rank"])
    # the slowest rank's time reaches every rank
    assert res[0]["t"] == res[1]["t"] == 3.0
    # each rank has its own batch, and each batch (and its verification) is reproducible
    assert res[0]["tokens"] != res[1]["tokens"]
    assert all(r["repeat_equal"] for r in res)
    assert all(min(r["out_len"]) >= 1 for r in res)
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_throughput(96, 20, 3.0, 2) == 2 * 96 * 20 / 3.0


def test_reference_arm_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    # the contract's keys, on the GPU arm's metric and workload
    for k in ("metric", "unit", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["metric"] == "verified tree tokens/s" and line["higher_is_better"] is True
    assert line["config"]["workload"] == "chain_g4_v1000_f32"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["unit"] == line["unit"]
    assert cb["cores"] >= 1 and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
