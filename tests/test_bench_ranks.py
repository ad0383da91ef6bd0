"""The replicas path of bench.py on CPU: two gloo ranks, each with its own
timing, agree on the slowest rank's time and on the whole-job value; the
reference arm prints on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]
        ms = bench.max_over_ranks(local_ms, world)
        q.put((rank, ms, bench.job_gbs(world, 2_000_000_000, ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [5.0, 5.0]
    # two replicas each streaming 2 GB in 5 ms: 800 GB/s for the job
    assert all(abs(o[2] - 800.0) < 1e-9 for o in out)


def test_single_rank_is_its_own_max():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert abs(bench.job_gbs(1, 10**9, 1.0) - 1000.0) < 1e-9


def test_reference_arm_prints_on_rank_zero_only():
    # rank 1 of a torchrun launch exits 0 without work and without output
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
