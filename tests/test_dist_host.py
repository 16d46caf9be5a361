"""Multi-rank host logic of bench.py on CPU with the gloo backend (world size 2):
environment parsing, the barrier and the max-over-ranks reduction that turn
per-rank device times into the reported number (weak scaling, no collective on
the data path)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    t = 10.0 + 5.0 * rank                      # per-rank timed region in ms
    m = bench.max_over_ranks(t, w, torch.device("cpu"))
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    results[rank] = m


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_barrier_gloo(world):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(results) == {0: 15.0, 1: 15.0}


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    bench.barrier(1)


def test_reference_arm_is_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])) == 0
    assert capsys.readouterr().out == ""
