"""One gloo rank of tests/test_multirank.py (run as a script: RANK WORLD PORT)."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path[:0] = [ROOT, os.path.join(ROOT, "tests")]

import numpy as np  # noqa: E402
import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402
import parity_util as PU  # noqa: E402
from speculative_decoding_draft_tree_gb300 import workloads as W  # noqa: E402


def _lists(rows):
    return [np.asarray(r).tolist() for r in rows]


def main():
    rank, world, port = int(sys.argv[1]), int(sys.argv[2]), int(sys.argv[3])
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = W.make_config(2, scale="small", device="cpu", seeds=bench.rank_seeds(rank))
    snap = PU.snapshot(w)
    orc = PU.oracle_verify(w, snap)
    w2 = W.make_config(2, scale="small", device="cpu", seeds=bench.rank_seeds(rank))
    again = PU.oracle_verify(w2, PU.snapshot(w2))
    t = bench.max_over_ranks(1.0 + 2.0 * rank, world)
    print(json.dumps(dict(rank=rank, t=t, tokens=snap["tokens"].tolist(),
                          out_len=np.asarray(orc["out_len"]).tolist(),
                          repeat_equal=_lists(orc["out_tokens"]) == _lists(again["out_tokens"]))))
    dist.barrier()
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
