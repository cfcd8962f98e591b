"""Sharding of the path over several GPUs (host logic).

Chunks are independent units: a chunk's scale, ring segments and outputs depend on that chunk
alone (the pipelined HCCL AllReduce article allreduces chunk by chunk, §3.1).  So a job split
over `world` GPUs gives each GPU a contiguous range of the chunk table; every GPU quantises and
reduces all W virtual ranks of its range, writing the disjoint range of outputs
[offsets[j0], offsets[j1]).  Passing the sub-table offsets[j0 : j1 + 1] (global element offsets,
no rebasing) to any of the library's calls does exactly that.  When every GPU needs the whole
output, one gather of the disjoint ranges follows; no other exchange is needed.
"""
import numpy as np


def shard_range(offsets, world, rank):
    """Contiguous chunk range [j0, j1) of `rank` out of `world`, balanced by elements: rank r
    starts at the first chunk boundary at or after r/world of the elements.  Ranges are disjoint,
    in rank order, and cover every chunk (a rank may get none)."""
    off = np.asarray(offsets, dtype=np.int64)
    nc = len(off) - 1
    if world < 1 or not 0 <= rank < world or nc < 0:
        raise ValueError("bad world / rank / table")
    total = int(off[-1] - off[0])

    def start(r):
        if r == 0:
            return 0
        if r >= world:
            return nc
        target = off[0] + (total * r + world - 1) // world
        return int(np.searchsorted(off[:nc], target, side="left"))

    return start(rank), start(rank + 1)


def shard_table(offsets, world, rank):
    """The rank's sub-table offsets[j0 : j1 + 1] (host int64) and its chunk count j1 - j0."""
    j0, j1 = shard_range(offsets, world, rank)
    off = np.asarray(offsets, dtype=np.int64)
    return off[j0:j1 + 1].copy(), j1 - j0


def gather_outputs(out, offsets, world, rank, group=None):
    """After every rank wrote its range of `out` (a 1-D float32 tensor of offsets[-1] elements,
    on any device the process group's backend takes), fill in the other ranks' ranges from them:
    one all_gather of equal-length (padded) pieces."""
    import torch
    import torch.distributed as dist
    off = np.asarray(offsets, dtype=np.int64)
    ranges = [shard_range(off, world, r) for r in range(world)]
    spans = [(int(off[a]), int(off[b])) for a, b in ranges]
    width = max(1, max(hi - lo for lo, hi in spans))
    lo, hi = spans[rank]
    mine = torch.zeros(width, dtype=out.dtype, device=out.device)
    mine[:hi - lo] = out[lo:hi]
    pieces = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(pieces, mine, group=group)
    for r, (a, b) in enumerate(spans):
        if r != rank and b > a:
            out[a:b] = pieces[r][:b - a]
    return out
