"""Window-range sharding over ranks (one process per GPU) on the CPU: the split, the
slicing of the input waveforms and the one sum of the statistics, with two gloo
ranks on 127.0.0.1 and the CPU oracle standing in for each rank's GPU."""
import multiprocessing as mp
import socket

import numpy as np
import pytest

import synth
from gate_level_logic_gb300 import shard


@pytest.mark.parametrize("W,world", [(256, 1), (256, 2), (256, 8), (10, 3), (7, 7), (4096, 6)])
def test_window_range_covers_every_window_once(W, world):
    got = [shard.window_range(W, world, r) for r in range(world)]
    assert got[0][0] == 0 and got[-1][1] == W
    assert all(a[1] == b[0] for a, b in zip(got, got[1:]))
    sizes = [b - a for a, b in got]
    assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1


def test_window_range_rejects():
    with pytest.raises(ValueError):
        shard.window_range(3, 4, 0)
    with pytest.raises(ValueError):
        shard.window_range(8, 2, 2)


@pytest.mark.parametrize("w0,w1", [(0, 16), (0, 1), (5, 9), (15, 16)])
def test_slice_equals_window_selection(w0, w1):
    _, stim = synth.make("50k")
    off, words = shard.slice_windows(stim.pi_off, stim.pi_words, stim.num_inputs, stim.num_windows, w0, w1)
    ref = synth.select_windows(stim, np.arange(w0, w1))
    assert np.array_equal(off, ref.pi_off) and np.array_equal(words, ref.pi_words)


def test_single_rank_sum_is_identity():
    tc, t1 = np.arange(5), np.arange(5) * 7
    a, b = shard.sum_stats(None, tc, t1)
    assert np.array_equal(a, tc) and np.array_equal(b, t1)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_ranks_sum_to_the_whole_run(oracle_lib):
    pytest.importorskip("torch.distributed")
    import multirank_worker
    net, stim = synth.make("50k")
    whole = oracle_lib.simulate(net, stim, threads=4)
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=multirank_worker.shard_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(queue.get(timeout=300) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [(g[1], g[2]) for g in got] == [(0, 8), (8, 16)]
    for g in got:
        assert np.array_equal(np.frombuffer(g[4], np.int64), whole.tc)
        assert np.array_equal(np.frombuffer(g[5], np.int64), whole.t1)
    assert all(p.exitcode == 0 for p in procs)
