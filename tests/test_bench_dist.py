"""The multi-replica host logic of bench.py on CPU: two ranks over gloo (127.0.0.1) reduce
their times to the slowest rank's and report the work of both over that time.  The path
has no data exchange (replicas only), so this reduction is the only collective."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    times = bench.slowest_rank([10.0 + rank, 5.0 - rank], dist, "cpu")
    queue.put((rank, times, bench.job_tflops(world, 1e12, 4, times[0])))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, times, tflops in results:
        assert times == [11.0, 5.0]                      # each entry: the slower rank's value
        assert tflops == pytest.approx(2 * 1e12 * 4 / 0.011 / 1e12)


def test_single_replica_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank([3.0, 1.5], None, "cpu") == [3.0, 1.5]
    assert bench.job_tflops(1, 2e12, 10, 1000.0) == pytest.approx(20.0)
