"""The seeded input generators: netlist structure, delay tables, stimulus format."""
import numpy as np
import pytest

import synth
from helpers import EOW, INF


@pytest.mark.parametrize("name", ["tiny", "50k"])
def test_netlist_is_levelised(name):
    net, _ = synth.make(name)
    P = net.num_inputs
    lo = net.level_offsets
    for lvl in range(net.num_levels):
        g0, g1 = lo[lvl], lo[lvl + 1]
        for g in range(g0, g1):
            pins = net.fanin_net[net.fanin_off[g]:net.fanin_off[g + 1]]
            assert len(pins) == net.type_num_pins[net.gate_type[g]]
            assert (pins < P + g0).all()                       # only earlier levels
            first = pins[0]
            assert (first < P) if lvl == 0 else (P + lo[lvl - 1] <= first < P + g0)


def test_impossible_arcs_follow_unateness():
    ok = synth.possible_rows(synth.truth_table("NAND2"), 2)
    # row = 4*pin + 2*e_in + e_out, RISE = 0, FALL = 1: NAND is negative unate
    assert ok.tolist() == [False, True, True, False] * 2
    assert synth.possible_rows(synth.truth_table("XOR2"), 2).all()
    assert synth.possible_rows(synth.truth_table("BUF"), 1).tolist() == [True, False, False, True]
    mux = synth.possible_rows(synth.truth_table("MUX2"), 3)
    assert mux[8:12].all()                                    # select pin is binate
    assert mux[0:4].tolist() == [True, False, False, True]    # data pins positive unate


def test_delay_tables_shape_and_conditions():
    net, _ = synth.make("50k")
    for g in range(0, net.num_gates, 97):
        ty = net.gate_type[g]
        n = int(net.type_num_pins[ty])
        D = net.dly_data[net.gate_dly_off[g]:net.gate_dly_off[g] + 4 * n * (1 << (n - 1))].reshape(4 * n, -1)
        tt = net.tt_data[net.type_tt_off[ty]:net.type_tt_off[ty] + (1 << n)]
        ok = synth.possible_rows(tt, n)
        assert (D[~ok] == INF).all()
        fin = D[ok]
        assert ((fin >= 5) & (fin <= 60)).all()
        if net.type_names[ty] not in ("AOI21", "MUX2"):
            assert (fin == fin[:, :1]).all()                  # unconditional: one value per row
    cond = [g for g in range(net.num_gates) if net.type_names[net.gate_type[g]] == "AOI21"][:50]
    varied = 0
    for g in cond:
        D = net.dly_data[net.gate_dly_off[g]:net.gate_dly_off[g] + 48].reshape(12, 4)
        varied += int((D[D[:, 0] != INF] != D[D[:, 0] != INF][:, :1]).any())
    assert varied > 40


def _check_format(w):
    w = np.asarray(w, np.int64)
    assert w[-1] == EOW
    head = 2 if w[0] == -1 else 1
    assert w[head - 1] == 0
    body = w[head:-1]
    assert (np.diff(np.concatenate(([0], body))) > 0).all()


def test_stimulus_format_and_windows():
    spec = synth.StimulusSpec(num_inputs=20, cycles=103, period=50, activity=0.3, windows=7, seed=3,
                              glitch_frac=0.5, glitch_span=(1, 5))
    st = synth.generate_stimulus(spec)
    assert st.window_cycles.tolist() == [15] * 5 + [14] * 2
    assert (st.window_len == st.window_cycles * 50).all()
    for p in range(20):
        prev_final = None
        for w in range(7):
            wave = st.window(p, w)
            _check_format(wave)
            assert (wave[:-1] < st.window_len[w]).all()
            init = 1 if wave[0] == -1 else 0
            if prev_final is not None:
                assert init == prev_final              # windows continue the same signal
            prev_final = (wave.size - 2) % 2
    sub = synth.select_windows(st, [6, 2])
    assert sub.num_windows == 2
    assert np.array_equal(sub.window(5, 0), st.window(5, 6))
    assert np.array_equal(sub.window(5, 1), st.window(5, 2))
    assert st.stats["glitch_pairs"] > 0


def test_generator_is_seeded():
    a_net, a_st = synth.make("tiny")
    b_net, b_st = synth.make("tiny")
    assert np.array_equal(a_net.fanin_net, b_net.fanin_net)
    assert np.array_equal(a_net.dly_data, b_net.dly_data)
    assert np.array_equal(a_st.pi_words, b_st.pi_words)
