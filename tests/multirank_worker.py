"""Rank body for the multi-process CPU tests (spawned, gloo backend)."""
import os
import sys


def bench_rank(rank: int, world: int, port: int, out_dir: str):
    import torch.distributed as dist

    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, rank, world)
        # each rank's own time; the job is timed by the slowest rank
        ms = 10.0 + 5.0 * rank
        bench.barrier(world)
        ms_max = bench.max_over_ranks(ms, world)
        rate = bench.job_rate(world, 1e9, 100, ms_max)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{ms_max} {rate}\n")
    finally:
        dist.destroy_process_group()
