"""Cycle windows spread over GPUs, one process per GPU.

The GATSPI page splits cycle parallelism over several GPUs (Section 5, the multi-GPU
paragraph and Fig. 6, where the kernel time behaves as T = T1 / N + c).  Windows are
independent re-simulations, so the split needs no exchange while simulating:

* every rank takes one contiguous range of the windows (``window_range``);
* every rank holds the whole netlist, its own pool and its own library context, and
  loads only its windows' input waveforms (``slice_windows``);
* the only collective is one sum over the ranks of the per-gate TC and T1 (int64) at
  the end (``sum_stats``); T0 follows from the total window time.

Nothing here simulates: each rank runs the CUDA library on its windows.
"""
from __future__ import annotations

import numpy as np


def window_range(num_windows: int, world: int, rank: int) -> tuple:
    """Contiguous windows [w0, w1) of ``rank`` among ``world`` ranks: every window once,
    in order, the ranges differing in size by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank %d of %d" % (rank, world))
    if num_windows < world:
        raise ValueError("%d windows cannot be spread over %d ranks" % (num_windows, world))
    return num_windows * rank // world, num_windows * (rank + 1) // world


def slice_windows(off, words, num_inputs: int, num_windows: int, w0: int, w1: int):
    """The input waveforms of windows [w0, w1) from a CSR over every (input, window),
    input-major and window-minor (the layout gatspi_load_waveforms takes): returns the
    CSR of the same layout over the range.  Each input's windows of the range are one
    contiguous run of the source."""
    off = np.asarray(off, np.int64)
    words = np.asarray(words, np.int32)
    W, n = num_windows, w1 - w0
    if not 0 <= w0 < w1 <= W or off.size != num_inputs * W + 1:
        raise ValueError("bad window range or offsets")
    rows = off[:-1].reshape(num_inputs, W)
    first = rows[:, w0]
    last = off[np.arange(num_inputs) * W + w1]
    runs = last - first
    base = np.zeros(num_inputs + 1, np.int64)
    base[1:] = np.cumsum(runs)
    src = np.repeat(first - base[:-1], runs) + np.arange(int(base[-1]))
    new_off = (off[:-1].reshape(num_inputs, W)[:, w0:w1] - first[:, None] + base[:-1, None]).ravel()
    return np.append(new_off, base[-1]), words[src]


def sum_stats(dist, tc, t1):
    """The per-gate TC and T1 summed over every rank (the run's one collective):
    int64 all-reduce over the default process group (on the GPU for NCCL, on the host
    for gloo).  ``dist`` None means a single rank."""
    tc = np.asarray(tc, np.int64)
    t1 = np.asarray(t1, np.int64)
    if dist is None:
        return tc.copy(), t1.copy()
    import torch
    both = torch.from_numpy(np.concatenate([tc, t1]))
    if dist.get_backend() == "nccl":
        both = both.cuda()
    dist.all_reduce(both, op=dist.ReduceOp.SUM)
    both = both.cpu().numpy()
    return both[:tc.size].copy(), both[tc.size:].copy()


class WindowShard:
    """One rank's share of a run: its windows' context on this rank's GPU."""

    def __init__(self, net, window_len, world: int, rank: int, pool_words: int, **kw):
        from .simulator import Simulator
        wl = np.asarray(window_len, np.int64).reshape(-1)
        self.num_windows = int(wl.size)
        self.num_inputs = int(net.num_inputs)
        self.w0, self.w1 = window_range(self.num_windows, world, rank)
        self.total_window_time = int(wl.sum())
        self.sim = Simulator(net, wl[self.w0:self.w1], pool_words=pool_words, **kw)

    def load(self, off, words, stream=None):
        """Load this rank's windows from the whole run's (input, window) CSR."""
        o, w = slice_windows(off, words, self.num_inputs, self.num_windows, self.w0, self.w1)
        self.sim.load(o, w, stream=stream)

    def simulate(self, stream=None):
        self.sim.simulate(stream=stream)

    def stats(self, dist=None):
        """(tc, t0, t1) of the whole run: this rank's statistics summed over the ranks."""
        tc, _, t1 = self.sim.toggle_stats()
        tc, t1 = sum_stats(dist, tc, t1)
        return tc, self.total_window_time - t1, t1

    def close(self):
        self.sim.close()
