"""Worker for the replicas test (launched by torch.distributed.run with the
gloo backend on CPU): every rank reduces its own timings with bench.py's
cross-replica helpers and writes what it got to <out_dir>/rank<r>.json."""
import json
import os
import sys

import torch
import torch.distributed as dist

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def main():
    out_dir = sys.argv[1]
    dist.init_process_group("gloo")
    rank, ws = dist.get_rank(), dist.get_world_size()
    got = bench._max_over_ranks([1.0 + rank, 10.0 - rank, 3.5], torch.device("cpu"))
    value = bench._whole_job_value(ws, 2e12, got[0])
    dist.barrier()
    # one file per rank: the ranks' stdout streams interleave
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"rank": rank, "ws": ws, "max": got, "value": value}, f)
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
