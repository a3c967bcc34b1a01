"""The multi-rank logic of bench.py on the CPU: world size 2 over gloo (the
timing aggregation the GPU ranks use over NCCL), and the reference arm's rank
rule under torchrun.  No GPU."""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, ms, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        got = bench.max_over_ranks(torch, ms[rank], dist, device="cpu")
        out.put((rank, got, bench.whole_job_gbs(world, 1_000_000, 10, got)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo():
    """Each rank times its own replica; the job's time is the slowest rank's,
    and the job's GB/s counts every rank's bytes over that time."""
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    world, port, ms = 2, _free_port(), [1.5, 2.0]
    procs = [ctx.Process(target=_rank, args=(r, world, port, ms, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(out.get(timeout=10) for _ in range(world))
    assert [r[1] for r in res] == [2.0, 2.0]
    # 2 ranks x 1 MB x 10 steps in 2 ms = 10 GB/s
    assert all(abs(r[2] - 10.0) < 1e-9 for r in res)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(torch, 3.25, None) == 3.25
    assert bench.whole_job_gbs(1, 81_592_320, 100, 2.7) == pytest.approx(3021.9, rel=1e-4)


def test_reference_arm_other_ranks_exit_quietly():
    """Under torchrun only rank 0 runs and prints the reference arm; the
    other ranks exit 0 without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
