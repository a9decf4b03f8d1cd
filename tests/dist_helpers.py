"""Worker functions for the multi-process (gloo, CPU) tests; importable by spawned children."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def max_over_ranks_worker(rank, ws, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    # rank r reports times (1 + r, 5 - r, 3): the job's times are the slowest rank's
    out = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 3.0], ws)
    results.put((rank, out))
    dist.barrier()
    dist.destroy_process_group()
