"""Small test helpers: building one-gate netlists and reading waveforms.

The value-at-time reading of a waveform follows the array format of the GATSPI
page (Fig. 3): entry k is the time from which the signal holds value k % 2.
"""
import numpy as np

import synth

EOW = int(synth.EOW)
INF = int(synth.INF)


def value_at(wave, t):
    """Logic value of a Fig. 3 waveform at time t (t >= 0)."""
    wave = np.asarray(wave)
    body = wave[:-1]
    k = int(np.searchsorted(body, t, side="right")) - 1
    return k % 2


def changes(wave):
    """Toggle timestamps (everything after the initial [0] / [-1, 0] head, before EOW)."""
    wave = [int(x) for x in wave]
    assert wave[-1] == EOW
    head = 2 if wave[0] == -1 else 1
    return wave[head:-1]


def single_gate(tt, n, delay_table, wire_rise=None, wire_fall=None, type_name="CELL"):
    """A netlist with n inputs feeding one gate."""
    wr = np.zeros(n, np.int32) if wire_rise is None else np.asarray(wire_rise, np.int32)
    wf = np.zeros(n, np.int32) if wire_fall is None else np.asarray(wire_fall, np.int32)
    return synth.build_netlist(num_inputs=n, level_gates=[1], type_names=[type_name], type_num_pins=[n],
                               type_tts=[tt], gate_type=[0], fanins=[list(range(n))], wire_rise=wr,
                               wire_fall=wf, delay_tables=[np.asarray(delay_table, np.int32)])


def uniform_delays(n, rise, fall, tt=None):
    """[4n][2**(n-1)] table with output-rise delay ``rise`` and output-fall delay ``fall``
    on every arc; arcs the truth table cannot exercise are INF when ``tt`` is given."""
    D = np.zeros((4 * n, 1 << (n - 1)), np.int64)
    for r in range(4 * n):
        D[r, :] = rise if r % 2 == 0 else fall
    if tt is not None:
        ok = synth.possible_rows(tt, n)
        D[~ok, :] = INF
    return D.astype(np.int32)


def permute_pin_weights(net, seed):
    """The same circuit with every gate's truth-table pin weights permuted at random
    and its truth table re-indexed to match (one cell type per gate)."""
    rng = np.random.default_rng(seed)
    G = net.num_gates
    tts, names, pins, weights = [], [], [], []
    for g in range(G):
        t = int(net.gate_type[g])
        n = int(net.type_num_pins[t])
        tt = net.tt_data[net.type_tt_off[t]:net.type_tt_off[t] + (1 << n)]
        wt = [1 << b for b in rng.permutation(n)]
        new = np.zeros(1 << n, np.uint8)
        for v in range(1 << n):                 # v: pin values, first pin most significant
            old_k = sum(((v >> (n - 1 - i)) & 1) << (n - 1 - i) for i in range(n))
            new_k = sum(((v >> (n - 1 - i)) & 1) * wt[i] for i in range(n))
            new[new_k] = tt[old_k]
        tts.append(new)
        names.append("%s_%d" % (net.type_names[t], g))
        pins.append(n)
        weights.extend(wt)
    out = synth.Netlist(
        num_inputs=net.num_inputs, num_gates=G, num_levels=net.num_levels, level_offsets=net.level_offsets,
        type_names=names, type_num_pins=np.array(pins, np.int32),
        type_tt_off=np.concatenate(([0], np.cumsum([len(t) for t in tts])[:-1])).astype(np.int32),
        tt_data=np.concatenate(tts).astype(np.uint8), gate_type=np.arange(G, dtype=np.int32),
        fanin_off=net.fanin_off, fanin_net=net.fanin_net, pin_weight=np.array(weights, np.int32),
        wire_rise=net.wire_rise, wire_fall=net.wire_fall, gate_dly_off=net.gate_dly_off, dly_data=net.dly_data)
    return out
