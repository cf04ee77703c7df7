"""The multi-rank host logic of bench.py on CPU, two gloo ranks.

The swap-in path partitions by request, so ranks own disjoint request blocks
and exchange nothing on the data path; only timing uses collectives (a
barrier, the max of the ranks' times, the sum of their work)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from hierarchical_kv_cache_hs_gb300 import tracegen as tg
        ops = bench.RankOps(dist, "cpu")
        ops.barrier()
        wl = tg.WORKLOADS["tiny_b1_c8k"].with_(B=3)
        reqs = bench.shard_requests(rank, wl.B)
        tr = tg.topk_trace(wl, steps=2, requests=reqs)
        q.put((rank, reqs, tr.sum(), ops.max(float(rank + 1)), ops.sum(float(10 * (rank + 1)))))
        ops.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_shard_requests_and_reduce_timing():
    from hierarchical_kv_cache_hs_gb300 import tracegen as tg
    tg.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, reqs0, s0, mx0, sm0), (r1, reqs1, s1, mx1, sm1) = got
    assert reqs0 == [0, 1, 2] and reqs1 == [3, 4, 5]
    assert not set(reqs0) & set(reqs1)
    assert s0 != s1  # different requests draw different traces
    assert mx0 == mx1 == 2.0
    assert sm0 == sm1 == 30.0


def test_single_process_ops_are_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    ops = bench.RankOps(None, "cpu")
    ops.barrier()
    assert ops.max(3.5) == 3.5 and ops.sum(2.0) == 2.0
    assert bench.shard_requests(0, 4) == [0, 1, 2, 3]
