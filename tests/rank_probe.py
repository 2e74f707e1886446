"""Stand-in for the benchmark's per-rank step, for the rank-launch test: each
rank joins the gloo process group through bench.py's helpers, reports a step
time of 1 + rank ms, and rank 0 prints one JSON line with the world size, the
ranks that took part and the max-over-ranks time."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import bench  # noqa: E402


def main():
    ws, rank, local = bench.dist_env()
    d = bench.init_dist(ws, "gloo")
    bench.barrier(d)
    seen = torch.zeros(ws, dtype=torch.int64)
    seen[rank] = 1
    if d is not None:
        d.all_reduce(seen)
    worst = bench.max_over_ranks(1.0 + rank, d)
    if rank == 0:
        print(json.dumps({"n_gpus": ws, "ranks": [i for i in range(ws) if seen[i]],
                          "local_ranks_ok": local == 0, "ms_per_step": worst,
                          "value": bench.whole_job_rate(1e9, ws, worst)}), flush=True)
    if d is not None:
        d.destroy_process_group()


if __name__ == "__main__":
    main()
