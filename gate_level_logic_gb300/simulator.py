"""A small Python front end over the C ABI: marshals numpy netlist arrays into the
C structs, allocates the waveform pool as a torch int32 CUDA tensor, and passes
torch streams through.  All simulation work happens in libgatspi.so.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import gatspi as _c


def _arr(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Simulator:
    """One netlist, one window configuration, one borrowed waveform pool.

    ``net`` is any object with the netlist arrays of include/gatspi.h as attributes
    (num_inputs, num_gates, num_levels, level_offsets, gate_type, type_num_pins,
    type_tt_off, tt_data, fanin_off, fanin_net, pin_weight, wire_rise, wire_fall,
    gate_dly_off, dly_data).  ``pulse_percent`` is PATHPULSEPERCENT, the inertial
    reject limit of the interconnect and gate filters as a percentage of the delay
    (100 = the GATSPI page's setting; 0 = transport delay).
    """

    def __init__(self, net, window_len, pool_words: int = None, pool=None, flags: int = 0,
                 device: int = None, pulse_percent: int = 100):
        import torch
        self._torch = torch
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        wl = _arr(window_len, np.int64).reshape(-1)
        self.num_windows = int(wl.size)
        self.num_inputs = int(net.num_inputs)
        self.num_gates = int(net.num_gates)
        self.num_levels = int(net.num_levels)
        self.num_nets = self.num_inputs + self.num_gates
        self._owns_pool = pool is None
        if pool is None:
            if pool_words is None:
                raise ValueError("give pool_words or pool")
            pool_words = (int(pool_words) + 3) // 4 * 4
            pool = torch.empty(pool_words, dtype=torch.int32, device=self.device)
        self.pool = pool
        keep = dict(
            level_offsets=_arr(net.level_offsets, np.int32), gate_type=_arr(net.gate_type, np.int32),
            type_num_pins=_arr(net.type_num_pins, np.int32), type_tt_off=_arr(net.type_tt_off, np.int32),
            tt_data=_arr(net.tt_data, np.uint8), fanin_off=_arr(net.fanin_off, np.int32),
            fanin_net=_arr(net.fanin_net, np.int32), pin_weight=_arr(net.pin_weight, np.int32),
            wire_rise=_arr(net.wire_rise, np.int32), wire_fall=_arr(net.wire_fall, np.int32),
            gate_dly_off=_arr(net.gate_dly_off, np.int64), dly_data=_arr(net.dly_data, np.int32),
            window_len=wl,
        )
        nl = _c.gatspi_netlist(
            self.num_inputs, self.num_gates, self.num_levels, len(keep["type_num_pins"]),
            keep["level_offsets"].ctypes.data, keep["gate_type"].ctypes.data, keep["type_num_pins"].ctypes.data,
            keep["type_tt_off"].ctypes.data, keep["tt_data"].size, keep["tt_data"].ctypes.data,
            keep["fanin_off"].ctypes.data, keep["fanin_net"].ctypes.data, keep["pin_weight"].ctypes.data,
            keep["wire_rise"].ctypes.data, keep["wire_fall"].ctypes.data, keep["gate_dly_off"].ctypes.data,
            keep["dly_data"].size, keep["dly_data"].ctypes.data)
        if int(pulse_percent) != 100:
            flags = int(flags) | _c.GATSPI_FLAG_PULSE_PERCENT
        cfg = _c.gatspi_config(self.num_windows, keep["window_len"].ctypes.data, int(flags), int(pulse_percent))
        self.pulse_percent = int(pulse_percent)
        with torch.cuda.device(self.device):
            self.ctx = _c.gatspi_create(nl, cfg, self.pool.data_ptr(), self.pool.numel())
        self.window_len = wl

    # -- lifecycle ---------------------------------------------------------------
    def close(self):
        """Release the context; a pool this object allocated is dropped with it."""
        if getattr(self, "ctx", None):
            _c.gatspi_destroy(self.ctx)
            self.ctx = None
            if getattr(self, "_owns_pool", False):
                self.pool = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -- calls -------------------------------------------------------------------
    def load(self, pi_off, pi_words, stream=None):
        """Load input waveforms from numpy (host) arrays or torch CUDA tensors."""
        torch = self._torch
        if isinstance(pi_words, torch.Tensor) and pi_words.is_cuda:
            off = pi_off.to(torch.int64).contiguous()
            words = pi_words.to(torch.int32).contiguous()
            _c.gatspi_load_waveforms(self.ctx, off.data_ptr(), words.data_ptr(), words.numel(), _c.GATSPI_DEVICE,
                                     _stream_handle(stream))
            return
        if isinstance(pi_words, torch.Tensor):
            off_a, words_a = pi_off.contiguous(), pi_words.contiguous()
            off_p, words_p, n = off_a.data_ptr(), words_a.data_ptr(), words_a.numel()
        else:
            off_a, words_a = _arr(pi_off, np.int64), _arr(pi_words, np.int32)
            off_p, words_p, n = off_a.ctypes.data, words_a.ctypes.data, words_a.size
        _c.gatspi_load_waveforms(self.ctx, off_p, words_p, n, _c.GATSPI_HOST, _stream_handle(stream))

    def load_testbench(self, tb_off, tb_words, stream=None):
        """Load whole-testbench input waveforms (one per input, times from the start of
        the testbench) and cut them into this simulator's windows on the GPU.  Numpy
        (host) arrays or torch tensors (host or CUDA)."""
        torch = self._torch
        if isinstance(tb_words, torch.Tensor) and tb_words.is_cuda:
            off = tb_off.to(device=tb_words.device, dtype=torch.int64).contiguous()
            words = tb_words.to(torch.int32).contiguous()
            _c.gatspi_load_testbench(self.ctx, off.data_ptr(), words.data_ptr(), words.numel(), _c.GATSPI_DEVICE,
                                     _stream_handle(stream))
            return
        if isinstance(tb_words, torch.Tensor):
            off_a, words_a = tb_off.contiguous(), tb_words.contiguous()
            off_p, words_p, n = off_a.data_ptr(), words_a.data_ptr(), words_a.numel()
        else:
            off_a, words_a = _arr(tb_off, np.int64), _arr(tb_words, np.int32)
            off_p, words_p, n = off_a.ctypes.data, words_a.ctypes.data, words_a.size
        _c.gatspi_load_testbench(self.ctx, off_p, words_p, n, _c.GATSPI_HOST, _stream_handle(stream))

    def simulate(self, stream=None):
        _c.gatspi_simulate(self.ctx, _stream_handle(stream))

    def sync(self):
        _c.gatspi_sync(self.ctx)

    def toggle_stats(self):
        """(tc, t0, t1) int64 arrays [num_gates], summed over windows."""
        tc = np.zeros(max(self.num_gates, 1), np.int64)
        t0 = np.zeros_like(tc)
        t1 = np.zeros_like(tc)
        _c.gatspi_toggle_stats(self.ctx, tc.ctypes.data, t0.ctypes.data, t1.ctypes.data)
        n = self.num_gates
        return tc[:n], t0[:n], t1[:n]

    def toggle_stats_view(self):
        """(tc, t1, sum of window lengths) without a copy: read-only uint64 views of
        the library's pinned host buffers, valid until the next simulate or close
        (t0 = sum of window lengths - t1)."""
        tcp, t1p, ws = _c.gatspi_toggle_stats_host(self.ctx)
        if self.num_gates == 0 or not tcp:
            empty = np.zeros(0, np.uint64)
            return empty, empty, ws
        u64 = ctypes.POINTER(ctypes.c_uint64)
        tc = np.ctypeslib.as_array(ctypes.cast(tcp, u64), shape=(self.num_gates,))
        t1 = np.ctypeslib.as_array(ctypes.cast(t1p, u64), shape=(self.num_gates,))
        tc.flags.writeable = False
        t1.flags.writeable = False
        return tc, t1, ws

    def waveform(self, net: int, window: int) -> np.ndarray:
        n = _c.gatspi_get_waveform(self.ctx, net, window, 0, 0)
        buf = np.zeros(max(n, 1), np.int32)
        _c.gatspi_get_waveform(self.ctx, net, window, buf.ctypes.data, buf.size)
        return buf[:n]

    def input_stats(self):
        """(tc, t0, t1) int64 arrays [num_inputs], summed over windows."""
        tc = np.zeros(max(self.num_inputs, 1), np.int64)
        t0 = np.zeros_like(tc)
        t1 = np.zeros_like(tc)
        _c.gatspi_input_stats(self.ctx, tc.ctypes.data, t0.ctypes.data, t1.ctypes.data)
        n = self.num_inputs
        return tc[:n], t0[:n], t1[:n]

    def write_saif(self, path, design: str = "top", timescale: str = "1 ps", net_names=None):
        """Write every net's statistics as a SAIF 2.0 file (names: n<index> unless given)."""
        if net_names is None:
            _c.gatspi_write_saif(self.ctx, str(path), design, timescale, 0)
            return
        names = [n.encode() for n in net_names]
        if len(names) != self.num_nets:
            raise ValueError("need one name per net (%d)" % self.num_nets)
        arr = (ctypes.c_char_p * len(names))(*names)
        _c.gatspi_write_saif(self.ctx, str(path), design, timescale, ctypes.addressof(arr))

    def export_offsets(self):
        """(start, length) of every (net, window) waveform in the pool, net-major."""
        n = self.num_nets * self.num_windows
        start = np.zeros(max(n, 1), np.int64)
        length = np.zeros(max(n, 1), np.int32)
        _c.gatspi_export_offsets(self.ctx, start.ctypes.data, length.ctypes.data, n)
        return start[:n], length[:n]

    def export_all(self):
        """(off, words): every (net, window) waveform gathered gap-free, net-major and
        window-minor, as CSR."""
        return self.export_windows(np.arange(self.num_windows))

    def export_windows(self, windows):
        """(off, words) CSR of the waveforms of the given windows for every net,
        net-major: waveform (net, windows[s]) is entry net * len(windows) + s."""
        sel = _arr(windows, np.int32).reshape(-1)
        off = np.zeros(self.num_nets * sel.size + 1, np.int64)
        _c.gatspi_export_windows(self.ctx, sel.ctypes.data, sel.size, off.ctypes.data, 0, 0)
        words = np.zeros(max(int(off[-1]), 1), np.int32)
        _c.gatspi_export_windows(self.ctx, sel.ctypes.data, sel.size, off.ctypes.data, words.ctypes.data, words.size)
        return off, words[:int(off[-1])]

    def lanes_per_window(self) -> int:
        """Lanes the next simulate gives each window (32 // W when windows are cut into
        time chunks, else 1)."""
        return _c.gatspi_lanes_per_window(self.ctx)

    def net_digests(self, net_begin: int = 0, num_nets: int = None, with_words: bool = False):
        """uint64 [num_nets]: the 64-bit FNV-1a digest of each net's waveforms in
        window order (gatspi_net_digests); with ``with_words`` also the int64 number
        of words of each net."""
        if num_nets is None:
            num_nets = self.num_nets - net_begin
        n = int(num_nets)
        out = np.zeros(max(n, 1), np.uint64)
        words = np.zeros(max(n, 1), np.int64)
        _c.gatspi_net_digests(self.ctx, int(net_begin), n, out.ctypes.data, words.ctypes.data)
        return (out[:n], words[:n]) if with_words else out[:n]

    def views(self) -> _c.gatspi_views:
        return _c.gatspi_device_views(self.ctx)

    def pool_used(self) -> int:
        return int(self.views().pool_used)

    def pool_host(self) -> np.ndarray:
        """Copy of the used part of the pool."""
        used = self.pool_used()
        return self.pool[:used].cpu().numpy()

    def set_level_timing(self, on: bool):
        """Record per-level kernel times in the following simulate calls (serialises
        the kernels), or stop recording them."""
        _c.gatspi_set_level_timing(self.ctx, on)

    def level_times(self):
        """(simulation-kernel ms, bounds-kernel ms) per level of the last simulate."""
        sim = np.zeros(max(self.num_levels, 1), np.float32)
        bnd = np.zeros_like(sim)
        _c.gatspi_level_times(self.ctx, sim.ctypes.data, bnd.ctypes.data, self.num_levels)
        return sim[:self.num_levels], bnd[:self.num_levels]
