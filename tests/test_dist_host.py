"""The N > 1 host path of bench.py on CPU: two gloo ranks, max over ranks and
the whole-job throughput formula (replicas, weak scaling)."""
import multiprocessing as mp
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r "took" 10 + 5r ms for its steps
        q.put((rank, bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 15.0, 1: 15.0}


def test_job_throughput_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    # two replicas, each 10 steps of 1e12 FLOP, slowest rank 20 ms -> 1000 TFLOP/s
    assert abs(bench.job_throughput(1e12, 10, 2, 20.0) - 1000.0) < 1e-9
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
