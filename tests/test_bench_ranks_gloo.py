"""The N > 1 host logic of bench.py on CPU: two gloo ranks, each with its own
time, agree on the slowest rank and on the whole-job throughput."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [2.0, 3.0][rank]
    e2e = [5.0, 4.0][rank]
    got = bench.max_over_ranks([ms, e2e])
    out[rank] = (got, bench.job_tflops(world, 1e12, got[0]))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_value():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        got, tflops = res[rank]
        assert got == [3.0, 5.0]
        assert tflops == pytest.approx(2 * 1e12 / 3e-3 / 1e12)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]


def _bench(args, env=None):
    import subprocess

    e = dict(os.environ)
    for key in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        e.pop(key, None)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, env=e,
                          capture_output=True, text=True, timeout=300)


def test_gpus_flag_launches_that_many_ranks():
    """`bench.py --gpus 2` without a launcher starts two ranks itself (gloo in
    this dry run), and rank 0 alone prints the line with n_gpus 2 and the
    slowest rank's time."""
    import json

    out = _bench(["--gpus", "2", "--dry-run", "--steps", "3", "--warmup", "3"])
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["ms_per_step"] == 2.0


def test_gpus_flag_must_match_the_launcher():
    out = _bench(["--gpus", "2", "--dry-run"], env={"WORLD_SIZE": "1", "RANK": "0", "LOCAL_RANK": "0"})
    assert out.returncode != 0 and "WORLD_SIZE" in out.stderr
    out = _bench(["--gpus", "1", "--dry-run"])
    assert out.returncode == 0 and '"n_gpus": 1' in out.stdout
