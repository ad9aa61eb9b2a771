"""The N>1 host logic of bench.py on CPU: two gloo ranks, each with its own step time and
workload, aggregate to the max step time and the summed bytes (weak scaling, no data-path
collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, gbps = bench.aggregate_ranks(1.0 + rank, 1_000_000_000, world, device="cpu")
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, ms, gbps))


def test_two_rank_aggregation_is_max_time_and_summed_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, ms, gbps in res:
        assert ms == pytest.approx(2.0)                   # max over ranks
        assert gbps == pytest.approx(2 * 1.0 / 2.0e-3)    # 2 GB over 2 ms = 1000 GB/s


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    ms, gbps = bench.aggregate_ranks(0.5, 1_000_000_000, 1)
    assert ms == 0.5 and gbps == pytest.approx(2000.0)
