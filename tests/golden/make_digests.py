"""Write the oracle's digests of the large workloads to ``tests/golden/digests/``.

These are the expected values of the full-size parity tests (``tests/test_gpu_digests.py``):
the 5M-gate workload, the scan-style 500k-gate run, all sixteen points of the
activity x windows sweep on the 1M-gate netlist, and three of them again below
PATHPULSEPERCENT 100 (names ending in -qN).  Each is simulated completely by
the CPU oracle (Algorithm 1 of the GATSPI page, Section 3), every gate in every
window, and stored as per-level records (exact word, TC and T1 sums plus
position-keyed mixes of every gate's waveform digest, TC and T1; see
``tests/digests.py``).  Windows are independent re-simulations, so long runs are
done in consecutive batches of windows with each net's digest carried over.

Only ``oracle/`` computes anything here; ``synth/`` draws the seeded inputs.

    python tests/golden/make_digests.py                 # every workload missing a file
    python tests/golden/make_digests.py sweep-0.05-256  # named ones (recomputed)
"""
from __future__ import annotations

import json
import os
import platform
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(HERE))

import digests  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402

OUT = os.path.join(HERE, "digests")
# (gate, window) tasks per batch: bounds the oracle's per-task tables (16 B each)
TASKS_PER_BATCH = 1 << 26


def compute(name, desc, make, threads):
    t0 = time.time()
    net, stim = make()
    t_gen = time.time() - t0
    W = stim.num_windows
    per = max(1, min(W, TASKS_PER_BATCH // max(net.num_inputs + net.num_gates, 1)))
    state = None
    t1 = time.time()
    batches = 0
    for w0 in range(0, W, per):
        sel = np.arange(w0, min(W, w0 + per))
        sub = stim if sel.size == W else synth.select_windows(stim, sel)
        state = oracle.digest(net, sub, state=state, threads=threads, pulse_percent=digests.pulse_percent(name))
        batches += 1
    t_sim = time.time() - t1
    rec = {
        "workload": name,
        "description": desc,
        "inputs_sha256": digests.inputs_sha256(net, stim),
        "num_inputs": int(net.num_inputs), "num_gates": int(net.num_gates), "num_levels": int(net.num_levels),
        "num_windows": int(W), "window_time": int(state.window_time),
        "pulse_percent": digests.pulse_percent(name),
        "events": int(state.tc.sum()), "words": int(state.net_words.sum()),
        "inputs": digests.input_record(net.num_inputs, state.net_hash, state.net_words),
        "levels": digests.level_records(net.level_offsets, net.num_inputs, state.net_hash, state.net_words,
                                        state.tc, state.t1),
        "oracle": {"threads": threads, "batches": batches, "seconds": round(t_sim, 1),
                   "generate_seconds": round(t_gen, 1), "machine": platform.machine()},
    }
    return rec


def main(argv):
    os.makedirs(OUT, exist_ok=True)
    threads = os.cpu_count() or 1
    table = digests.large_workloads()
    names = argv or [n for n in table if not os.path.exists(os.path.join(OUT, n + ".json"))]
    oracle.build()
    for name in names:
        desc, make = table[name]
        rec = compute(name, desc, make, threads)
        path = os.path.join(OUT, name + ".json")
        with open(path + ".tmp", "w") as f:
            json.dump(rec, f, indent=1)
            f.write("\n")
        os.replace(path + ".tmp", path)
        print("%s: %d events, %d words, %.0f s" % (name, rec["events"], rec["words"], rec["oracle"]["seconds"]),
              flush=True)


if __name__ == "__main__":
    main(sys.argv[1:])
