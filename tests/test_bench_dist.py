"""The benchmark's multi-rank path on CPU: two gloo ranks, replica batches,
slowest-rank time and summed bytes (no collective on the data path)."""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    from paged_kv_cache_140_gb300 import workloads as W
    w, r, lr = bench.dist_env()
    assert (w, r, lr) == (world, rank, rank)
    bench.dist_init("gloo")
    # Each rank builds its own replica batch from a rank-offset seed.
    cfg = W.CONFIGS["7b"]
    b = W.make_batch("7b", num_seqs=3, seed=140000 + cfg["number"] + 1000 * rank)
    ms, units = bench.aggregate(1.0 + rank, float(bench.kv_bytes(b)), world)
    tot = [None] * world
    dist.all_gather_object(tot, bench.kv_bytes(b))
    q.put((rank, ms, units, sum(tot), b.context_lens.tolist()))
    dist.destroy_process_group()


def test_two_rank_gloo_aggregation():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    assert all(r[1] == 2.0 for r in res)               # slowest rank's time
    assert res[0][2] == res[1][2] == res[0][3]          # bytes of both replicas
    assert res[0][4] != res[1][4]                       # distinct replica batches


def test_single_rank_aggregate_is_identity():
    import bench
    assert bench.aggregate(3.5, 42.0, 1) == (3.5, 42.0)


def test_byte_accounting_matches_definition():
    import numpy as np

    import bench
    from paged_kv_cache_140_gb300 import workloads as W
    b = W.make_batch("13b", num_seqs=7)
    assert bench.kv_bytes(b) == int(b.context_lens.sum()) * 40 * 128 * 2 * 2
    # A single partition longer than every context: no split partials.
    base = bench.decode_bytes(b, 4096)
    q = o = 7 * 40 * 128 * 2
    tables = int(np.ceil(b.context_lens / 16).sum()) * 4 * 40
    assert base == bench.kv_bytes(b) + q + o + tables + 7 * 4
    assert bench.decode_bytes(b, 16) > base
