"""The benchmark's multi-rank bookkeeping (replicas, one per GPU), on CPU with two gloo ranks:
the reported time is the slowest rank's and the value counts every rank's work."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_secs = 2.0 if rank == 1 else 1.0            # rank 1 is the slow one
        secs, value = bench.whole_job(my_secs, 1e12, 10, world, dist, torch.device("cpu"))
        out[rank] = (secs, value)
    finally:
        dist.destroy_process_group()


def test_whole_job_uses_slowest_rank_and_all_work():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        secs, value = res[rank]
        assert secs == 2.0                              # the max over ranks
        assert value == pytest.approx(1e12 * 10 * world / 2.0 / 1e12)


def test_whole_job_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    secs, value = bench.whole_job(0.5, 2e12, 4, 1, None, torch.device("cpu"))
    assert secs == 0.5 and value == pytest.approx(16.0)


# ---- `bench.py --gpus N` with no launcher: the script starts the replica ranks itself -------

def _cpu_run_ours(args, rank, world, local_rank, dist):
    # CPU stand-in for the GPU work of one replica, with the benchmark's own bookkeeping
    import json
    import bench
    secs, value = bench.whole_job(1.0 + rank, 1e12, args.steps, world, dist, torch.device("cpu"))
    with open(os.path.join(os.environ["BENCH_TEST_OUT"], f"rank{rank}.json"), "w") as fh:
        json.dump({"rank": rank, "world": world, "local_rank": local_rank, "secs": secs,
                   "value": value, "backend": dist.get_backend() if dist else None}, fh)


def _replica_child(local_rank, argv, world, port):
    sys.path.insert(0, ROOT)
    import bench
    bench.run_ours = _cpu_run_ours
    bench._replica_main(local_rank, argv, world, port)


def test_launch_replicas_runs_every_rank_through_the_benchmark_path(tmp_path, monkeypatch):
    import json
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("BENCH_TEST_OUT", str(tmp_path))
    for var in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(var, raising=False)
    bench.launch_replicas(["--gpus", "2", "--steps", "5"], 2, target=_replica_child)
    res = [json.loads((tmp_path / f"rank{r}.json").read_text()) for r in range(2)]
    for r, d in enumerate(res):
        assert d["rank"] == r and d["local_rank"] == r and d["world"] == 2
        assert d["backend"] == "gloo"
        assert d["secs"] == 2.0                          # the slowest rank's time
        assert d["value"] == pytest.approx(1e12 * 5 * 2 / 2.0 / 1e12)


def test_gpus_flag_without_launcher_reports_the_rank_count():
    # the reference arm through the real command line: two replica processes, one line
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
