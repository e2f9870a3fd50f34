"""The N > 1 host logic of bench.py on CPU: two gloo ranks (processes) reduce
their per-rank timings with the same helper the GPU run uses (max over ranks:
replicas finish when the slowest does) and the job rate counts the units of
every rank. Also: under torchrun, only rank 0 of the reference arm prints."""
import multiprocessing
import os
import socket
import subprocess
import sys

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        per = {"mask": 0.1 * (rank + 1), "fwd": 1.2 - 0.1 * rank, "bwd": 4.0 + rank, "total": 10.0 + rank}
        out = bench.reduce_max(per, world, "cpu")
        rate = bench.job_rate(100.0, world, out["fwd"])
        q.put((rank, out, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_rank():
    ctx = multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, out, rate in res:
        assert out == {"mask": 0.2, "fwd": 1.2, "bwd": 5.0, "total": 11.0}
        assert abs(rate - 2 * 100.0 / 1.2e-3) < 1e-6  # both ranks' units over the slowest time


def test_single_rank_keeps_its_timings():
    sys.path.insert(0, ROOT)
    import bench
    per = {"fwd": 1.5, "bwd": 4.5}
    assert bench.reduce_max(per, 1, None) == per
    assert bench.job_rate(3.0, 1, 2.0) == 1500.0


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference"], env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
    # fewer than 3 warm-up steps are refused
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"], capture_output=True,
                       text=True, timeout=120)
    assert r.returncode != 0 and "warm-up" in r.stderr
