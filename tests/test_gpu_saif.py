"""Statistics out of the CUDA path: the TC/T1 copied to the host level by level during
the simulation, the inputs' statistics, and the SAIF file that carries them.

The inputs' statistics are pinned through the oracle: a zero-delay buffer on every
input reproduces its waveform, so the oracle's TC/T1 of those buffers are the
inputs' own.
"""
import os
import re

import numpy as np
import pytest

import synth
from helpers import uniform_delays
from test_gpu_parity import THREADS, gpu, pool_for, run_gpu  # noqa: F401  (gpu is a fixture)

pytestmark = pytest.mark.gpu


def _buffers_on_inputs(P):
    tt = synth.truth_table("BUF")
    return synth.build_netlist(num_inputs=P, level_gates=[P], type_names=["BUF"], type_num_pins=[1], type_tts=[tt],
                               gate_type=[0] * P, fanins=[[p] for p in range(P)], wire_rise=np.zeros(P),
                               wire_fall=np.zeros(P), delay_tables=[uniform_delays(1, 0, 0, tt)] * P)


@pytest.mark.parametrize("name", ["tiny", "50k"])
def test_input_stats(gpu, oracle_lib, name):
    _, stim = synth.make(name)
    tb = synth.testbench(name)
    net = _buffers_on_inputs(stim.num_inputs)
    ref = oracle_lib.simulate(net, stim)
    for use_tb in (False, True):
        with gpu(net, stim.window_len, pool_words=pool_for(ref, net) + 2 * tb.words.size
                 + 3 * stim.num_windows * stim.num_inputs) as sim:
            if use_tb:
                sim.load_testbench(tb.off, tb.words)
            else:
                sim.load(stim.pi_off, stim.pi_words)
            tc, t0, t1 = sim.input_stats()
            assert np.array_equal(tc, ref.tc) and np.array_equal(t1, ref.t1) and np.array_equal(t0, ref.t0)


@pytest.mark.parametrize("flags", [0, 1, 2])
def test_statistics_on_every_launch_path(gpu, oracle_lib, flags):
    """Graph replay, direct launches and timed launches all dump TC/T1 the same way;
    a second simulate refreshes them."""
    net, stim = synth.make("50k")
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    with gpu(net, stim.window_len, pool_words=pool_for(ref, net), flags=flags) as sim:
        sim.load(stim.pi_off, stim.pi_words)
        for _ in range(2):
            sim.simulate()
            tc, t0, t1 = sim.toggle_stats()
            assert np.array_equal(tc, ref.tc) and np.array_equal(t1, ref.t1) and np.array_equal(t0, ref.t0)


def _parse_saif(text):
    tokens = re.findall(r'\(|\)|"[^"]*"|(?:\\.|[^\s()\\])+', text)
    pos = 0

    def expr():
        nonlocal pos
        if tokens[pos] == "(":
            pos += 1
            out = []
            while tokens[pos] != ")":
                out.append(expr())
            pos += 1
            return out
        tok = tokens[pos]
        pos += 1
        return tok

    tree = expr()
    assert pos == len(tokens)
    return tree


def test_saif_file(gpu, oracle_lib, tmp_path):
    net, stim = synth.make("50k")
    ref = oracle_lib.simulate(net, stim, threads=THREADS)
    with gpu(net, stim.window_len, pool_words=pool_for(ref, net)) as sim:
        sim.load(stim.pi_off, stim.pi_words)
        sim.simulate()
        path = os.path.join(tmp_path, "run.saif")
        sim.write_saif(path, design="dut", timescale="1 ps")
        itc, _, it1 = sim.input_stats()
        text = open(path).read()
    tree = _parse_saif(text)
    assert tree[0] == "SAIFILE"
    fields = {item[0]: item[1:] for item in tree[1:] if isinstance(item, list)}
    duration = int(fields["DURATION"][0])
    assert duration == int(stim.window_len.sum())
    assert fields["TIMESCALE"] == ["1", "ps"] and fields["DESIGN"] == ['"dut"']
    inst = fields["INSTANCE"]
    assert inst[0] == "dut" and inst[1][0] == "NET"
    nets = inst[1][1:]
    P = net.num_inputs
    assert len(nets) == P + net.num_gates
    for k, entry in enumerate(nets):
        assert entry[0] == "n%d" % k
        vals = {f[0]: int(f[1]) for f in entry[1:]}
        tc, t1 = (itc[k], it1[k]) if k < P else (ref.tc[k - P], ref.t1[k - P])
        assert vals == {"T0": duration - t1, "T1": t1, "TX": 0, "TC": tc, "IG": 0}, k


def test_saif_names_are_escaped(gpu, oracle_lib, tmp_path):
    net, stim = synth.make("tiny")
    ref = oracle_lib.simulate(net, stim)
    names = ["in[%d]" % p for p in range(net.num_inputs)] + ["u%d/y" % g for g in range(net.num_gates)]
    with gpu(net, stim.window_len, pool_words=pool_for(ref, net)) as sim:
        sim.load(stim.pi_off, stim.pi_words)
        sim.simulate()
        path = os.path.join(tmp_path, "named.saif")
        sim.write_saif(path, net_names=names)
        text = open(path).read()
    assert "(in\\[0\\]" in text and "(u3\\/y" in text
    nets = _parse_saif(text)[-1][2][1:]
    assert [n[0] for n in nets][:2] == ["in\\[0\\]", "in\\[1\\]"]
    assert int(dict((f[0], f[1]) for f in nets[net.num_inputs + 3][1:])["TC"]) == ref.tc[3]
