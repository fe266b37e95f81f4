"""The N > 1 path of bench.py on CPU: two gloo ranks (no GPU).

The step has no cross-request exchange, so N GPUs run N independent replicas; the only
collective is the aggregation of the timed region (slowest rank's time, all ranks' tokens).
These tests run that aggregation over a real two-process gloo group, and check that the
reference arm leaves every rank but 0 without work."""
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


def _rank_main(rank: int, world: int, port: int, out) -> None:
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench  # the benchmark's own aggregation
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: timed-region durations (r + 1) ms and 10 (r + 1) ms, tokens 100 (r + 1) and 7
        times, counts = bench.aggregate_over_ranks([rank + 1.0, 10.0 * (rank + 1)], [100 * (rank + 1), 7],
                                                   torch.device("cpu"))
        dist.barrier()
        out.put((rank, times, counts))
    finally:
        dist.destroy_process_group()


def test_aggregation_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, times, counts in got:
        assert times == [2.0, 20.0]        # the slowest rank's durations
        assert counts == [300.0, 14.0]     # tokens of all ranks
    # whole-job throughput: all ranks' tokens over the slowest rank's time
    assert got[0][2][0] / (got[0][1][0] * 1e-3) == pytest.approx(150_000.0)


def test_aggregation_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.aggregate_over_ranks([1.5, 2.5], [3, 4], torch.device("cpu")) == ([1.5, 2.5], [3.0, 4.0])


def test_reference_arm_other_ranks_do_no_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=120, env=env)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
