"""Multi-rank host logic of bench.py on CPU with the gloo backend (world size 2):
environment parsing, the barrier and the max-over-ranks reduction that turn
per-rank device times into the reported number (weak scaling, no collective on
the data path)."""
import json
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
    assert bench.run_reference(bench.parse_args(["--impl", "reference", "--gpus", "2", "--steps", "1",
                                                 "--warmup", "0"])) == 0
    assert capsys.readouterr().out == ""


_RANK_SCRIPT = r'''
import json, os, sys, time
sys.path.insert(0, %(root)r)
import torch
import bench

class WallTimer:
    def start(self):
        self.t0 = time.perf_counter()
    def stop(self):
        self.t1 = time.perf_counter()
    def elapsed_ms(self):
        return (self.t1 - self.t0) * 1e3

args = bench.parse_args(sys.argv[1:])
rank, world, local = bench.dist_env()
bench.check_world(args, world)
bench.dist_init(world, "gloo")
calls = []
def step(i):                       # the CPU stand-in for one step: rank r takes (r + 1) * 20 ms
    calls.append(i)
    time.sleep(0.02 * (rank + 1))
ms = bench.run_timed(step, args.steps, world, torch.device("cpu"), WallTimer(), lambda: None)
assert calls == list(range(args.steps))
if rank == 0:
    print(json.dumps({"n_gpus": world, "steps": args.steps, "ms_per_step": ms}), flush=True)
import torch.distributed as dist
dist.destroy_process_group()
'''


def test_gpus_flag_relaunches_one_rank_per_gpu(monkeypatch):
    """bench.py --gpus N started without a launcher re-runs itself as N ranks."""
    import bench
    seen = {}
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench, "launch_ranks", lambda n, argv, script=None: seen.update(n=n, argv=argv) or 0)
    assert bench.main(["--gpus", "4", "--steps", "3", "--warmup", "3"]) == 0
    assert seen == {"n": 4, "argv": ["--gpus", "4", "--steps", "3", "--warmup", "3"]}


def test_world_must_match_gpus(monkeypatch):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit):
        bench.check_world(bench.parse_args(["--gpus", "4"]), 2)
    bench.check_world(bench.parse_args(["--gpus", "2"]), 2)


def test_two_ranks_timed_region_max_over_ranks(tmp_path):
    """Two gloo ranks launched by bench.launch_ranks (torch.distributed.run, as `bench.py --gpus 2`
    does) run the GPU arms' timed region (bench.run_timed: barrier, sync, timer, steps, sync,
    barrier, max over ranks) around a CPU stand-in step; rank 0 alone prints n_gpus 2 and the
    slower rank's time per step."""
    import subprocess
    import sys

    import bench
    script = tmp_path / "rank.py"
    script.write_text(_RANK_SCRIPT % {"root": bench.ROOT})
    cmd = [sys.executable, "-c", "import sys, bench; sys.exit(bench.launch_ranks(2, %r, script=%r))"
           % (["--gpus", "2", "--steps", "5"], str(script))]
    env = dict(os.environ, PYTHONPATH=bench.ROOT)
    env.pop("WORLD_SIZE", None)
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env, cwd=bench.ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    assert lines[0]["n_gpus"] == 2 and lines[0]["steps"] == 5
    assert 38.0 <= lines[0]["ms_per_step"] < 80.0   # rank 1's 40 ms steps, not rank 0's 20 ms
