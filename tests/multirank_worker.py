"""Worker of the two-rank CPU test: runs bench.py's rank reductions over gloo."""
import os


def reduce_worker(rank, world, port, queue):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    r, w, local = bench._dist()
    dist = bench._init_pg(w)
    try:
        bench._barrier(dist)
        slowest = bench._max_over_ranks(dist, 1.5 + r)       # per-rank time: the job takes the slowest
        total = bench._sum_over_ranks(dist, 10.0 * (r + 1))  # per-rank events: the job sums them
        bench._barrier(dist)
        queue.put((r, w, local, slowest, total))
    finally:
        dist.destroy_process_group()
