"""The multi-GPU split (host logic), on the CPU: chunk ranges per rank, and a world-size-2 gloo
run where each process reduces its range of a multi-bucket table (with the oracle, standing in for
a GPU) and the gathered output matches the unsplit result bit for bit."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import __graft_entry__

__graft_entry__.build()  # the package loads libgq.so on import (it has no fallback)
from dp_gradient_bucket_gb300 import shard


def _table(seed, nb=6):
    rng = np.random.default_rng(seed)
    import oracle
    buckets = [int(x) for x in rng.integers(0, 300000, nb)] + [0, 5]
    return buckets, oracle.plan_chunks(buckets, 4)


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8, 13])
def test_ranges_partition_the_table(world):
    for seed in range(5):
        _, off = _table(seed)
        nc = len(off) - 1
        ranges = [shard.shard_range(off, world, r) for r in range(world)]
        assert ranges[0][0] == 0 and ranges[-1][1] == nc
        for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
            assert a0 <= a1 == b0 <= b1
        # balance: no rank's elements exceed its share by more than one chunk
        total = int(off[-1])
        biggest = int(np.diff(off).max()) if nc else 0
        for a, b in ranges:
            assert int(off[b] - off[a]) <= -(-total // world) + biggest


def test_rejects_bad_arguments():
    off = np.array([0, 4, 8])
    with pytest.raises(ValueError):
        shard.shard_range(off, 0, 0)
    with pytest.raises(ValueError):
        shard.shard_range(off, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        import workloads as wl
        W = 4
        buckets, off = _table(11)
        n = int(off[-1])
        stride = -(-n // 4) * 4
        rows = np.zeros(W * stride, dtype=np.float32)
        for r in range(W):
            wl.fill(2, r, 0, n, rows[r * stride:r * stride + n])
        sub, k = shard.shard_table(off, world, rank)
        out = torch.zeros(n, dtype=torch.float32)
        if k:
            codes, scales, _ = oracle.quantize(rows, W, stride, sub)
            part = oracle.reduce(codes, scales, W, stride, sub, oracle.RING)
            lo, hi = int(sub[0]), int(sub[-1])
            out[lo:hi] = torch.from_numpy(part[lo:hi])
        shard.gather_outputs(out, off, world, rank)
        want = oracle.fused(rows, W, stride, off, oracle.RING)[0]
        q.put((rank, bool(np.array_equal(out.numpy().view(np.uint32), want.view(np.uint32)))))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_gloo_split_matches_unsplit(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(world))
    assert res == {r: True for r in range(world)}
