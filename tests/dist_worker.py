"""Worker for the multi-rank CPU tests (spawned once per gloo rank; no GPU)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def bench_ranks(rank: int, world: int, port: int, queue) -> None:
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, world)   # the higher ranks are slower
        rate = bench.job_rate(world, 16384, ms)
        dist.barrier()
        queue.put((rank, ms, rate))
    finally:
        dist.destroy_process_group()
