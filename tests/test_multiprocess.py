"""The multi-rank host logic of bench.py on CPU with the gloo backend and two
ranks: the slowest rank's time is what every rank reports, the whole-job rate
counts every rank's units, and the reference arm runs on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r measured a step of 1.0 + r ms and a main kernel of 0.5 + 0.25 r ms
        got = bench.reduce_max_over_ranks([1.0 + rank, 0.5 + 0.25 * rank])
        out.put((rank, got, bench.job_rate(100.0, world, got[0])))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_with_two_gloo_ranks():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, rate in res:
        assert got == [2.0, 0.75]
        assert rate == pytest.approx(100.0 * 2 / 2.0e-3)


def test_single_process_reduce_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_max_over_ranks([3.0, 1.5]) == [3.0, 1.5]


def test_reference_arm_runs_on_rank_zero_only():
    """A non-zero rank of the reference arm exits 0 at once without output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
