"""The bench's multi-rank host logic on CPU with two gloo ranks: the job time is
the slowest rank's on every rank, the whole-job rate counts every rank's work,
and the reference arm runs on rank 0 only."""
import importlib.util
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


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = _bench()
        ms = 10.0 + 5.0 * rank                 # rank 1 is the slow one
        job_ms = bench.max_over_ranks(ms, world, torch.device("cpu"))
        out[rank] = (job_ms, bench.job_rate(100.0, job_ms, world))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_and_rate():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0           # the slowest rank's time, on both ranks
    assert res[0][1] == res[1][1] == pytest.approx(100.0 * 2 / 15e-3)


def test_single_rank_is_unchanged():
    bench = _bench()
    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    assert bench.job_rate(8.0, 2.0, 1) == pytest.approx(4000.0)


def test_reference_arm_other_ranks_do_nothing(capsys, monkeypatch):
    bench = _bench()
    monkeypatch.setenv("RANK", "1")

    class Args:
        config, steps, warmup, gpus = "tiny", 1, 0, 2
    assert bench.run_reference(Args) == 0
    assert capsys.readouterr().out == ""
