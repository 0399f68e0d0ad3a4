"""The multi-rank path of bench.py on CPU: two gloo ranks, max-over-ranks timing and the
weak-scaling (replica) throughput. No GPU: ranks exchange host tensors only."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r reports step times (r + 1, 10 - r): the job's times are the element-wise max
        got = bench.max_over_ranks([rank + 1.0, 10.0 - rank])
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_weak_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == [2.0, 10.0] and res[1] == [2.0, 10.0]
    sys.path.insert(0, ROOT)
    import bench
    # 2 replicas x 16384 tokens in 4 ms (the slowest rank) = 8.192e6 tokens/s
    assert abs(bench.weak_scaling_value(16384, 2, 4.0) - 8.192e6) < 1e-3
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]   # single process: identity
