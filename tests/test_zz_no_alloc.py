"""The allocation-free entry point gatspi_simulate_level_static.

It serves callers that cannot allocate device memory (for example code running
under a framework that owns all of the device memory, or code that must not
allocate after start-up): they hand over every buffer, and the level kernel's only
scratch sits in a fixed device array inside the library.  This test plays such a
caller: it allocates every buffer itself (torch tensors), lays out the input
waveforms and their window index itself, runs every logic level through the new
entry point, and checks the result against the regular path (gatspi_simulate) and
against the CPU oracle bit for bit -- twice in a row, since every call reuses the
one scratch array.
"""
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def _kernel_tables(net):
    """The delay tables in the layout gatspi_level_args documents: Fig. 4's row
    4*i + 2*e_in + e_out, column c at ((2*i + e_out) << n) | v, v = all pin values."""
    out = np.array(net.dly_data, np.int32)
    for g in range(net.num_gates):
        n = int(net.type_num_pins[net.gate_type[g]])
        cols = 1 << (n - 1)
        off = int(net.gate_dly_off[g])
        src = np.asarray(net.dly_data[off:off + 4 * n * cols])
        for i in range(n):
            b = n - 1 - i
            for e_out in (0, 1):
                for v in range(1 << n):
                    e_in = 0 if (v >> b) & 1 else 1
                    col = ((v >> (b + 1)) << b) | (v & ((1 << b) - 1))
                    out[off + (((2 * i + e_out) << n) | v)] = src[(4 * i + 2 * e_in + e_out) * cols + col]
    return out


def _pack(net):
    """The library's gate records (layout of gatspi_level_args): per gate the
    descriptor, the source net of every pin and every pin's wire delays."""
    G = net.num_gates
    n = net.type_num_pins[net.gate_type].astype(np.int64)
    mask = np.zeros(G, np.int64)
    for t in range(len(net.type_num_pins)):
        nt = int(net.type_num_pins[t])
        bits = sum(int(net.tt_data[net.type_tt_off[t] + k]) << k for k in range(1 << nt))
        mask[net.gate_type == t] = bits
    gd = np.zeros((G, 12), np.int64)
    gd[:, 1] = n | (mask << 8)
    gd[:, 2] = net.gate_dly_off & 0xFFFFFFFF
    gd[:, 3] = net.gate_dly_off >> 32
    wires = net.wire_rise.astype(np.int64) | (net.wire_fall.astype(np.int64) << 16)
    for i in range(4):
        has = n > i
        e = net.fanin_off[:-1][has] + i
        gd[has, 4 + i] = net.fanin_net[e]
        gd[has, 8 + i] = wires[e]
    return gd.astype(np.uint32).view(np.int32).ravel()


class Caller:
    """Owns every buffer; runs levels through the allocation-free entry point."""

    def __init__(self, net, stim, pool_words, pulse_percent=100):
        import torch
        from gate_level_logic_gb300 import gatspi
        self.gatspi, self.torch = gatspi, torch
        self.net, self.stim = net, stim
        P, G, W = net.num_inputs, net.num_gates, stim.num_windows
        self.N, self.W, self.nch = P + G, W, (W + 31) // 32
        dev = torch.device("cuda", 0)
        self.gate_desc = torch.from_numpy(_pack(net)).to(dev)
        self.dly = torch.from_numpy(_kernel_tables(net)).to(dev)
        self.window_len = torch.from_numpy(np.ascontiguousarray(stim.window_len, np.int32)).to(dev)
        self.pool = torch.zeros(pool_words, dtype=torch.int32, device=dev)
        self.net_base = torch.zeros(self.N, dtype=torch.int64, device=dev)
        self.wstart = torch.zeros(self.N * W, dtype=torch.int32, device=dev)
        self.wend = torch.zeros(self.N * W, dtype=torch.int32, device=dev)
        W4 = (W + 3) // 4 * 4
        self.wlen8 = torch.zeros(self.N * W4, dtype=torch.uint8, device=dev)
        most = int(np.diff(net.level_offsets).max()) if net.num_levels else 1
        self.perm = torch.zeros(max(most * W, 1), dtype=torch.int16, device=dev)
        self.goff = torch.zeros(max(most * (self.nch + 1), 1), dtype=torch.int32, device=dev)
        self.tc = torch.zeros(G, dtype=torch.int64, device=dev)
        self.t1 = torch.zeros(G, dtype=torch.int64, device=dev)
        self.level_base = torch.zeros(2, dtype=torch.int64, device=dev)
        self.pulse_percent = pulse_percent
        # input waveforms at the front of the pool, with their window index: each
        # input's windows back to back from its base
        off = stim.pi_off
        nw = int(off[-1])
        self.pool[:nw] = torch.from_numpy(np.ascontiguousarray(stim.pi_words, np.int32)).to(dev)
        k = np.arange(P * W)
        first = off[(k // W) * W]
        self.net_base[:P] = torch.from_numpy(np.ascontiguousarray(off[np.arange(P) * W], np.int64)).to(dev)
        self.wstart[:P * W] = torch.from_numpy((off[k] - first).astype(np.int32)).to(dev)
        self.wend[:P * W] = torch.from_numpy((off[k + 1] - first).astype(np.int32)).to(dev)
        l8 = np.zeros((P, W4), np.uint8)
        l8[:, :W] = np.minimum(off[k + 1] - off[k], 255).reshape(P, W)
        self.wlen8[:P * W4] = torch.from_numpy(l8.ravel()).to(dev)
        self.inputs_words = nw

    def args(self, gate_begin, num_gates, pool_words=None):
        g = self.gatspi
        return g.gatspi_level_args(
            self.gate_desc.data_ptr(), self.dly.data_ptr(), self.window_len.data_ptr(),
            self.pool.data_ptr(), self.pool.numel() if pool_words is None else pool_words,
            self.net_base.data_ptr(), self.wstart.data_ptr(), self.wend.data_ptr(), self.wlen8.data_ptr(),
            self.perm.data_ptr(),
            self.goff.data_ptr(), self.tc.data_ptr(), self.t1.data_ptr(),
            self.level_base.data_ptr(), self.net.num_inputs, self.W, gate_begin, num_gates,
            g.GATSPI_FLAG_PULSE_PERCENT, self.pulse_percent)

    def run(self, gaps=None, host_pool=True):
        """Every level, in order; returns (offsets, pool, tc, t1) as host arrays (the pool
        stays on the device unless host_pool).  gaps: {level: words left unused before
        the level's outputs}."""
        torch, g = self.torch, self.gatspi
        self.tc.zero_()
        self.t1.zero_()
        base = self.inputs_words
        lo = self.net.level_offsets
        stream = torch.cuda.current_stream().cuda_stream
        for lvl in range(self.net.num_levels):
            base += (gaps or {}).get(lvl, 0)
            self.level_base[0] = base
            g.gatspi_simulate_level_static(self.args(int(lo[lvl]), int(lo[lvl + 1] - lo[lvl])), stream)
            base = int(self.level_base[1].item())
        nb = self.net_base.cpu().numpy()
        ws = self.wstart.cpu().numpy().astype(np.uint32).astype(np.int64)
        we = self.wend.cpu().numpy().astype(np.uint32).astype(np.int64)
        k = np.arange(self.N * self.W)
        start = nb[k // self.W] + ws
        length = we - ws
        pool = self.pool[:base].cpu().numpy() if host_pool else self.pool
        return (start, length, base), pool, self.tc.cpu().numpy(), self.t1.cpu().numpy()


def _regular(net, stim, pool_words, pulse_percent=100):
    from gate_level_logic_gb300 import Simulator
    with Simulator(net, stim.window_len, pool_words=pool_words, pulse_percent=pulse_percent) as sim:
        sim.load(stim.pi_off, stim.pi_words)
        sim.simulate()
        tc, _, t1 = sim.toggle_stats()
        start, length = sim.export_offsets()
        used = sim.pool_used()
        return (start, length, used), sim.pool_host(), tc, t1


def _same_index(a, b):
    return np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2] == b[2]


def _gather(pool, index):
    """Every waveform's words, in (net, window) order (the gaps between output regions
    hold whatever the buffer held before and are not compared)."""
    start, length = np.asarray(index[0], np.int64), np.asarray(index[1], np.int64)
    first = np.concatenate(([0], np.cumsum(length)[:-1]))
    pos = np.repeat(start - first, length) + np.arange(int(length.sum()))
    return pool[pos]


@pytest.fixture(scope="module")
def built():
    import torch
    assert torch.cuda.is_available(), "needs a CUDA device"
    torch.cuda.set_device(0)
    from gate_level_logic_gb300 import build
    build.build()


@pytest.mark.parametrize("name,q", [("tiny", 100), ("50k", 100), ("tiny", 30), ("w256", 100), ("w256", 60)])
def test_static_levels_match_regular_path(built, oracle_lib, name, q):
    if name == "w256":     # eight chunks per gate
        net = synth.generate_netlist(synth.NetlistSpec(num_gates=800, num_inputs=20, num_levels=5, seed=5))
        stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=20, cycles=512, period=300, activity=0.4,
                                                          windows=256, seed=5, glitch_frac=0.3))
    else:
        net, stim = synth.make(name)
    pool_words = 1 << 26            # room for the bound-sized output regions of every level
    ref = _regular(net, stim, pool_words, pulse_percent=q)
    # the CPU oracle directly as well: every waveform in (net, window) order and the
    # statistics, so a fault shared by both GPU paths cannot pass unseen
    orc = oracle_lib.simulate(net, stim, threads=8, pulse_percent=q)
    caller = Caller(net, stim, pool_words, pulse_percent=q)
    for attempt in range(2):                        # two runs in a row share the scratch
        index, pool, tc, t1 = caller.run()
        assert _same_index(index, ref[0]), "waveform positions differ (run %d)" % attempt
        assert np.array_equal(_gather(pool, index), _gather(ref[1], ref[0])), "waveforms differ (run %d)" % attempt
        assert np.array_equal(tc, ref[2]) and np.array_equal(t1, ref[3]), "statistics differ (run %d)" % attempt
        assert np.array_equal(_gather(pool, index), orc.pool), "waveforms differ from the oracle (run %d)" % attempt
        assert np.array_equal(np.asarray(index[1], np.int64), np.diff(orc.off)), "lengths differ from the oracle"
        assert np.array_equal(tc, orc.tc) and np.array_equal(t1, orc.t1), "statistics differ from the oracle"


def test_sources_far_apart(built):
    """The inputs at the front of a pool of more than 2^32 words, the first level's
    outputs beyond word 2^32: gates of the next levels read sources that far apart,
    which offsets from one pointer cannot span in 32 bits, so those lanes count each
    pin's offsets from its own window.  Every waveform and statistic still equals the
    regular path's."""
    import torch
    net = synth.generate_netlist(synth.NetlistSpec(num_gates=600, num_inputs=16, num_levels=4, seed=9))
    stim = synth.generate_stimulus(synth.StimulusSpec(num_inputs=16, cycles=300, period=300, activity=0.4,
                                                      windows=40, seed=9, glitch_frac=0.3))
    lo, P, fo = np.asarray(net.level_offsets), net.num_inputs, net.fanin_off
    mixed = [g for g in range(lo[1], lo[2]) if (net.fanin_net[fo[g]:fo[g + 1]] < P).any()
             and (net.fanin_net[fo[g]:fo[g + 1]] >= P).any()]
    assert len(mixed) > 5
    gap = 1 << 32
    ref = _regular(net, stim, 1 << 24)
    caller = Caller(net, stim, gap + (1 << 24))
    index, pool, tc, t1 = caller.run(gaps={0: gap}, host_pool=False)
    assert int(index[0][P * stim.num_windows:].max()) > gap           # the outputs do sit beyond 2^32
    start, length = np.asarray(index[0], np.int64), np.asarray(index[1], np.int64)
    first = np.concatenate(([0], np.cumsum(length)[:-1]))
    pos = np.repeat(start - first, length) + np.arange(int(length.sum()))
    got = pool[torch.from_numpy(pos).to(pool.device)].cpu().numpy()
    assert np.array_equal(got, _gather(ref[1], ref[0]))
    assert np.array_equal(tc, ref[2]) and np.array_equal(t1, ref[3])
    del caller, pool
    torch.cuda.empty_cache()


def test_static_errors_and_limits(built):
    from gate_level_logic_gb300 import GatspiError, gatspi
    net, stim = synth.make("tiny")
    caller = Caller(net, stim, 1 << 20)
    lo = net.level_offsets
    # a pool too small for the first level: reported, and the next call starts clean
    caller.level_base[0] = caller.inputs_words
    with pytest.raises(GatspiError) as e:
        gatspi.gatspi_simulate_level_static(caller.args(0, int(lo[1]), pool_words=caller.inputs_words + 8))
    assert e.value.name == "GATSPI_EPOOL_OVERFLOW"
    ref = _regular(net, stim, 1 << 20)
    index, pool, tc, t1 = caller.run()
    assert _same_index(index, ref[0]) and np.array_equal(tc, ref[2])
    assert np.array_equal(_gather(pool, index), _gather(ref[1], ref[0]))
    # a level beyond the fixed scratch is refused before anything runs: one
    # look-back flag per 1024 gates, and 2^25 gates > 8192 x 1024
    assert stim.num_windows == 1
    big = caller.args(0, 1 << 25)
    with pytest.raises(GatspiError) as e:
        gatspi.gatspi_simulate_level_static(big)
    assert e.value.name == "GATSPI_EINVAL"
    assert ctypes.sizeof(gatspi.gatspi_level_args) > 0
