"""Body of one gloo rank for the multi-rank host-logic tests (CPU only)."""

import json
import os


def rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import torch.distributed as dist

    import bench
    import workloads

    r, w, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        # the slowest rank sets the time; the rate counts every rank's steps
        seconds = [0.5, 2.0, 1.0, 0.25][rank]
        slowest, rate = bench.job_rate(10, seconds, w)
        bench.barrier(w)
        rec = {
            "env": [r, w, local],
            "max": bench.reduce_max(float(rank * 3 + 1), w),
            "job": [slowest, rate],
            "sum": bench.sum_over_ranks(rank + 3, w),
            "seed": bench.rank_seed(r),
        }
        wl = workloads.make_workload("tiny", device="cpu", gen_device="cpu", seed=bench.rank_seed(r))
        rec["q_sum"] = float(wl.q.float().sum())
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump(rec, f)
    finally:
        dist.destroy_process_group()
