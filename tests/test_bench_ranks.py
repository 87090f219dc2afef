"""The bench's multi-rank host logic on CPU: two gloo ranks, the job time is the slowest
rank's, the job rate counts every rank's steps, and only rank 0 of the reference arm
prints."""
import importlib.util
import json
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    b = _bench()
    ms = 10.0 + 15.0 * rank                     # rank 1 is the slow one
    got = b.max_over_ranks(ms, world, torch.device("cpu"))
    out[rank] = (got, b.job_rate(world, 200, got))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 25.0
    assert res[0][1] == pytest.approx(2 * 200 / 0.025)


def test_single_rank_is_the_identity():
    b = _bench()
    assert b.max_over_ranks(12.5, 1, None) == 12.5
    assert b.job_rate(1, 10, 20.0) == pytest.approx(500.0)


def test_reference_arm_prints_on_rank_zero_only(capsys, monkeypatch):
    b = _bench()
    monkeypatch.setenv("RANK", "1")
    import sys
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--config", "single", "--steps", "1",
                                      "--warmup", "0"])
    assert b.main() == 0
    assert capsys.readouterr().out.strip() == ""
    monkeypatch.setenv("RANK", "0")
    assert b.main() == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_line_keeps_the_contract(capsys, monkeypatch):
    """Every key of the JSON line, with the reference arm's own cpu_baseline and e2e."""
    b = _bench()
    monkeypatch.setenv("RANK", "0")
    import sys
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--config", "single", "--steps", "2",
                                      "--warmup", "1"])
    assert b.main() == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert key in line, key
    assert line["metric"] == b.METRIC and line["unit"] == "steps/s" and line["higher_is_better"] is True
    assert line["steps"] == 2 and line["warmup"] == 1 and line["n_gpus"] == 1
    assert line["scaling"] == "weak" and line["vs_baseline"] is None and line["dtype"] == "f64"
    # a step is a timed sample of the batch step: ms_per_step is what the run spent per step
    # (the steps fit in the run's own wall time), value scales it to the whole batch
    assert line["full_step_ms"] == pytest.approx(1e3 / line["value"])
    assert line["sample_fraction"] == pytest.approx(line["ms_per_step"] / line["full_step_ms"])
    assert 0 < line["sample_fraction"] < 1
    assert line["steps"] * line["ms_per_step"] <= line["wall_s"] * 1e3 * 1.001
    assert line["config"]["workload"].startswith("single:")
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    assert cb["cpu"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == "steps/s"
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
