"""Window-range sharding on the GPU: the ranks of a split run, simulated one after the
other on cuda:0 (each its own context over its contiguous windows, as each would run
on its own GPU), give together exactly the oracle's whole run -- every (net, window)
waveform and the per-gate TC, T0 and T1 summed over the ranks."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def built():
    import torch
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    torch.cuda.set_device(0)
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("world", [2, 3, 16])
def test_split_ranks_equal_the_whole_run(built, oracle_lib, world):
    from gate_level_logic_gb300 import shard
    net, stim = synth.make("50k")
    whole = oracle_lib.simulate(net, stim, threads=8)
    P, G, W = net.num_inputs, net.num_gates, stim.num_windows
    tc = np.zeros(G, np.int64)
    t1 = np.zeros(G, np.int64)
    lens = np.zeros((P + G, W), np.int64)
    waves = {}
    for rank in range(world):
        part = shard.WindowShard(net, stim.window_len, world, rank, pool_words=4 * whole.pool.size + 4096)
        try:
            part.load(stim.pi_off, stim.pi_words)
            part.simulate()
            rtc, rt0, rt1 = part.stats()          # one rank alone: no collective
            assert np.array_equal(rt0 + rt1, np.full(G, int(stim.window_len.sum())))
            off, words = part.sim.export_all()
            w0, w1 = part.w0, part.w1
        finally:
            part.close()
        tc += rtc
        t1 += rt1
        n = w1 - w0
        lens[:, w0:w1] = np.diff(off).reshape(P + G, n)
        for net_id in range(P + G):
            for j in range(n):
                k = net_id * n + j
                waves[(net_id, w0 + j)] = words[off[k]:off[k + 1]]
    assert np.array_equal(tc, whole.tc) and np.array_equal(t1, whole.t1)
    assert np.array_equal(lens.ravel(), np.diff(whole.off))
    got = np.concatenate([waves[(k // W, k % W)] for k in range((P + G) * W)])
    assert np.array_equal(got, whole.pool)
