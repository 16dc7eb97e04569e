"""The bench's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1, as torchrun
launches them (one process per GPU; each rank simulates its own replica and only the
timing and event counts are reduced), and the reference arm's rank rule."""
import multiprocessing as mp
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_rank_reductions():
    pytest.importorskip("torch.distributed")
    import multirank_worker
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=multirank_worker.reduce_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(queue.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [g[0] for g in got] == [0, 1] and all(g[1] == 2 for g in got) and [g[2] for g in got] == [0, 1]
    assert all(g[3] == 2.5 for g in got)      # max over ranks of 1.5 + rank
    assert all(g[4] == 30.0 for g in got)     # sum over ranks of 10 * (rank + 1)
    assert all(p.exitcode == 0 for p in procs)


def test_single_rank_needs_no_group(monkeypatch):
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    rank, world, local = bench._dist()
    assert (rank, world, local) == (0, 1, 0)
    assert bench._init_pg(world) is None
    assert bench._max_over_ranks(None, 3.0) == 3.0 and bench._sum_over_ranks(None, 4.0) == 4.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import argparse
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(steps=1, warmup=0, pulse_percent=100)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""      # the other ranks exit without work or output


def test_kernel_hash_ignores_comments():
    import bench
    a = "int x = 1;  // one\n\n// a comment line\nint y = 2;\n"
    b = "int x = 1;\nint y = 2;   // two\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only("int x = 1;\n") != bench._code_only("int x = 2;\n")


def test_reference_arm_line(monkeypatch, capsys):
    """Rank 0 of the reference arm prints one JSON line on the bench's metric, unit and
    workload: the oracle timed as it stands on host cores, with its cpu_baseline block
    and an end-to-end block that copies nothing, both equal to the line's value."""
    import argparse
    import json
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    args = argparse.Namespace(steps=1, warmup=0, pulse_percent=100)
    assert bench.run_reference(args) == 0
    lines = [x for x in capsys.readouterr().out.splitlines() if x.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True and d["n_gpus"] == 1
    assert (d["steps"], d["warmup"]) == (1, 0) and d["ms_per_step"] > 0
    assert d["config"]["workload"] == bench.WORKLOAD_NAMES[bench.WORKLOAD]
    assert d["config"]["gates"] == 1_000_000 and d["config"]["windows"] == 256
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and "windows" in cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
