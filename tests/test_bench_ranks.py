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
