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


def shard_worker(rank, world, port, queue):
    """One rank of a window-sharded run on the CPU: the oracle stands in for the GPU on
    this rank's contiguous windows; the per-gate statistics are summed over gloo."""
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import numpy as np
    import torch.distributed as dist

    import oracle
    import synth
    from gate_level_logic_gb300 import shard
    dist.init_process_group("gloo")
    try:
        net, stim = synth.make("50k")
        w0, w1 = shard.window_range(stim.num_windows, world, rank)
        off, words = shard.slice_windows(stim.pi_off, stim.pi_words, net.num_inputs, stim.num_windows, w0, w1)
        part = synth.Stimulus(num_inputs=net.num_inputs, num_windows=w1 - w0, window_len=stim.window_len[w0:w1],
                              window_cycles=stim.window_cycles[w0:w1], pi_off=off, pi_words=words, stats={})
        r = oracle.simulate(net, part, threads=2)
        tc, t1 = shard.sum_stats(dist, r.tc, r.t1)
        queue.put((rank, w0, w1, int(np.asarray(tc, np.int64).sum()), tc.tobytes(), t1.tobytes()))
    finally:
        dist.destroy_process_group()
