"""Multi-rank host logic on CPU (gloo, world size 2): sequence sharding and the
max-over-ranks timing reduction the benchmark uses.  No GPU, no data-path
collective (the path itself exchanges nothing between ranks)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from bit_quantized_kv_02_gb300 import dist as kdist


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    r, w = kdist.init("gloo")
    lo, hi = kdist.shard(13, r, w)
    t = kdist.max_over_ranks(1.0 + r)
    s = kdist.sum_over_ranks(hi - lo)
    kdist.barrier()
    q.put((r, lo, hi, t, s))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_shard_partition():
    for total in (0, 1, 7, 64):
        for world in (1, 2, 3, 8):
            parts = [kdist.shard(total, r, world) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == total
            assert all(parts[i][1] == parts[i + 1][0] for i in range(world - 1))
            sizes = [b - a for a, b in parts]
            assert max(sizes) - min(sizes) <= 1


def test_gloo_two_ranks_max_and_sum():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1:3] for r in res] == [(0, 7), (7, 13)]
    assert all(r[3] == 2.0 for r in res)  # max over ranks of 1+rank
    assert all(r[4] == 13 for r in res)
