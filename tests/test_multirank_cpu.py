"""The N>1 path on CPU: replicas share nothing but the timing reduction.

bench.py runs one replica per rank; the only collectives are a barrier and
the max-over-ranks of the timed region (plus the sum of the units).  These
tests run that reduction with the gloo backend, world size 2, on the host."""
import importlib.util
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench = _bench()
    ms, units = bench.aggregate_over_ranks(1.5 + rank, 10.0 * (rank + 1))
    dist.barrier()
    out[rank] = (ms, units)
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert out[0] == out[1] == (2.5, 30.0)   # max time, summed units


def test_aggregate_without_process_group_is_identity():
    assert _bench().aggregate_over_ranks(3.0, 7.0) == (3.0, 7.0)


def test_reference_arm_prints_on_rank_zero_only(monkeypatch, capsys):
    bench = _bench()
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    class A:
        steps, warmup, config = 1, 3, "tiny"
    bench.run_reference(A())
    assert capsys.readouterr().out == ""
