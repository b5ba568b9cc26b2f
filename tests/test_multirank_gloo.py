"""Multi-rank host logic of the benchmark on CPU: 2 gloo ranks (no GPU).

Each rank runs an independent batch of the same shape (weak scaling, no
collective on the data path); the step time is the max over ranks and the
aggregate rate counts all ranks' bytes.
"""

import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from paged_kv_cache_55_gb300 import workloads as W
        seed = bench.rank_seed(0, rank)
        w = W.tiny_decode(seed=seed)
        acct = bench.step_accounting(w)
        my_ms = [3.0, 5.0][rank]
        mx = bench.reduce_max(my_ms)
        tot = bench.reduce_sum(float(acct["step_bytes"]))
        rate = bench.aggregate_rate(tot, mx * 1e-3)
        q.put((rank, seed, float(w.q[0, 0, 0]), mx, tot, rate, acct["step_bytes"]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_reduce():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, q0, mx0, tot0, rate0, b0), (r1, s1, q1, mx1, tot1, rate1, b1) = res
    assert s0 != s1, "ranks must draw independent batches"
    assert mx0 == mx1 == 5.0, "step time is the max over ranks"
    assert tot0 == tot1 == b0 + b1, "the aggregate counts every rank's bytes"
    assert np.isclose(rate0, (b0 + b1) / 5e-3)


def test_single_process_reductions_are_identity():
    import bench
    assert bench.reduce_max(2.5) == 2.5
    assert bench.reduce_sum(7.0) == 7.0
    assert bench.rank_seed(3, 0) == 3
