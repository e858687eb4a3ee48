"""The multi-GPU path of the benchmark, on the CPU with gloo: the path shards
into independent replicas (prefill by (batch, head), decode by request) with
no data-path exchange, so the process group only carries the barriers around
the timed region and the max over ranks of its time; the whole-job value is
units per rank x ranks / the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist, r, w, local = bench.dist_setup(backend="gloo")
    assert (r, w, local) == (rank, ws, rank)
    bench.barrier(dist)
    slowest = bench.max_over_ranks(dist, 10.0 + rank, "cpu")  # rank r "took" 10 + r ms
    out[rank] = (slowest, bench.aggregate(1000, w, slowest))
    bench.barrier(dist)
    dist.destroy_process_group()


@pytest.mark.parametrize("ws", [2, 3])
def test_replicas_take_the_slowest_rank(ws):
    out = mp.get_context("spawn").Manager().dict()  # no fork of a multi-threaded process
    mp.spawn(_worker, args=(ws, _free_port(), out), nprocs=ws, join=True)
    for rank in range(ws):
        slowest, value = out[rank]
        assert slowest == 10.0 + ws - 1
        assert value == pytest.approx(1000 * ws / ((10.0 + ws - 1) / 1e3))


def test_single_process_needs_no_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    dist, rank, ws, local = bench.dist_setup(backend="gloo")
    assert dist is None and (rank, ws, local) == (0, 1, 0)
    assert bench.max_over_ranks(None, 3.5, "cpu") == 3.5
    assert bench.aggregate(4096, 1, 2.0) == pytest.approx(4096 / 2e-3)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup = 1, 3
    bench.run_reference(A())
    assert capsys.readouterr().out == ""
