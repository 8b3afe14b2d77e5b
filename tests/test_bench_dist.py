"""The bench's multi-rank host logic on CPU: world_size 2 over gloo.

Each rank of `bench.py --gpus N` runs the whole workload on its own GPU (weak
scaling, no collective on the data path); the host side only needs a barrier
around the timed region and the maximum of the per-rank times. Both are
checked here with two gloo ranks, plus the reference arm's rule that only
rank 0 runs the oracle.
"""
import json
import multiprocessing as mp
import os
import socket

import pytest

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    d = bench.Dist(backend="gloo")
    try:
        d.barrier()
        slowest = d.max(1.5 + rank)          # this rank's "ms per step"
        d.barrier()
        out.put((rank, d.world, slowest))
    finally:
        d.close()


def test_two_gloo_ranks_barrier_and_max():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(out.get(timeout=5) for _ in procs)
    assert got == [(0, 2, 2.5), (1, 2, 2.5)]


def test_single_process_dist_is_identity(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    d = bench.Dist()
    assert d.world == 1 and d.rank == 0
    assert d.max(3.25) == 3.25
    d.barrier()
    d.close()


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    called = []
    monkeypatch.setattr(bench, "run_reference", lambda *a, **k: called.append(a))
    bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"])
    assert called == [] and capsys.readouterr().out == ""
    monkeypatch.setenv("RANK", "0")
    bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"])
    assert len(called) == 1


def test_reference_arm_json_line(monkeypatch, capsys):
    """The reference arm (the float64 oracle on sampled rows) prints one JSON
    line with the keys the bench contract asks of it."""
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    bench.main(["--impl", "reference", "--workload", "tiny_causal_bf16", "--steps", "2",
                "--warmup", "3", "--ref-seconds", "1.0"])
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["dtype"] == "f64"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "tiny_causal_bf16"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
