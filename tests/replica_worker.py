"""One rank of the replica-timing test (run as a subprocess by
test_replicas_cpu.py): joins a gloo group over 127.0.0.1, reports its rank
from the environment, the max-over-ranks of a rank-dependent time and the
whole-job rate bench.py would print."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402


def main():
    ws, rank, local = bench._dist()
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=ws)
    ms = 10.0 + 5.0 * rank           # this rank's timed window
    ms_max = bench.max_over_ranks(ms)
    rate = bench.job_rate(100, ws, ms_max)
    dist.barrier()
    dist.destroy_process_group()
    print(json.dumps({"ws": ws, "rank": rank, "local": local, "ms_max": ms_max, "rate": rate}))


if __name__ == "__main__":
    main()
