"""Child of test_multirank.py, launched by torch.distributed.run with the gloo
backend on the CPU: exercises bench.py's multi-rank host logic."""

import json
import os
import sys

import torch
import torch.distributed as dist

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from speculative_decoding_verification_13_gb300 import workloads  # noqa: E402


def main():
    out_dir = sys.argv[1]
    dist.init_process_group("gloo")
    ws, rank = dist.get_world_size(), dist.get_rank()
    # the slowest rank's time is the step time
    got = bench.max_over_ranks(1.5 + rank, dist, torch.device("cpu"))
    # every rank verifies its own independently seeded batch (no data exchange)
    b = workloads.make_batch("c1", "t1", device="cpu", seed_offset=rank)
    digest = float(b.target.double().sum())
    res = {"rank": rank, "ws": ws, "max": got, "digest": digest}
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)
    dist.barrier()
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
