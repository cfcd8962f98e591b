"""The oracle against the hand-derived worked cases in tests/golden/ (each file cites the
passage and shows the derivation of every expected value)."""
import numpy as np
import pytest

import _golden as G


def test_dynamic_chunk_sizes(orc):
    for n, eb, count, piece in G.chunk_sizes():
        assert orc.bucket_chunks(n, eb) == (count, piece), (n, eb)
        off = orc.plan_chunks([n], eb)
        assert len(off) == count + 1 and off[0] == 0 and off[-1] == n
        if n:
            assert np.all(np.diff(off)[:-1] == piece) and 0 < off[-1] - off[-2] <= piece


@pytest.mark.parametrize("name,case", G.keyed_cases("quantize_cases.txt"))
def test_quantize_cases(orc, name, case):
    g = np.array([G.f32(t) for t in case["grads"]], dtype=np.float32)
    off = np.array([int(t) for t in case["offsets"]], dtype=np.int64)
    codes, scales, nf = orc.quantize(g, 1, len(g), off)
    assert nf == 0
    assert [int(x) for x in codes] == [int(t) for t in case["codes"]], name
    want = [G.f32_bits(t) for t in case["scales"]]
    assert [int(x) for x in scales.reshape(-1).view(np.uint32)] == want, name


def test_unscale_f16(orc):
    (name, case), = G.keyed_cases("unscale_f16.txt")
    h = np.array([int(t, 16) for t in case["halves"]], dtype=np.uint16).view(np.float16)
    off = np.array([int(t) for t in case["offsets"]], dtype=np.int64)
    codes, scales, nf = orc.quantize(h, 1, len(h), off, loss_scale=float(case["loss_scale"][0]))
    assert nf == 0
    assert [int(x) for x in codes] == [int(t) for t in case["codes"]]
    assert int(scales.reshape(-1).view(np.uint32)[0]) == G.f32_bits(case["scales"][0])


def test_reduce_orders(orc):
    (name, case), = G.keyed_cases("reduce_orders.txt")
    W = int(case["W"][0])
    rows = [np.array([G.f32(t) for t in case["rank%d" % r]], dtype=np.float32) for r in range(W)]
    n = len(rows[0])
    grads = np.concatenate(rows)
    off = np.array([int(t) for t in case["offsets"]], dtype=np.int64)
    codes, scales, nf = orc.quantize(grads, W, n, off)
    assert [int(x) for x in scales.reshape(-1).view(np.uint32)] == [G.f32_bits(t) for t in case["scales"]]
    for order, key in ((orc.SEQ, "seq"), (orc.RING, "ring"), (orc.TREE, "tree")):
        out = orc.reduce(codes, scales, W, n, off, order)
        assert [int(x) for x in out.view(np.uint32)] == [G.f32_bits(t) for t in case[key]], key


def test_reduce_hier(orc):
    (name, case), = G.keyed_cases("reduce_hier.txt")
    W = int(case["W"][0])
    rows = [np.array([G.f32(t) for t in case["rank%d" % r]], dtype=np.float32) for r in range(W)]
    n = len(rows[0])
    grads = np.concatenate(rows)
    off = np.array([int(t) for t in case["offsets"]], dtype=np.int64)
    codes, scales, nf = orc.quantize(grads, W, n, off)
    assert [int(x) for x in scales.reshape(-1).view(np.uint32)] == [G.f32_bits(t) for t in case["scales"]]
    orders = [(orc.SEQ, "seq"), (orc.RING, "ring"), (orc.TREE, "tree")]
    orders += [(orc.HIER(L), "hier%d" % L) for L in (1, 2, 3, 6)]
    for order, key in orders:
        out = orc.reduce(codes, scales, W, n, off, order)
        assert [int(x) for x in out.view(np.uint32)] == [G.f32_bits(t) for t in case[key]], key


def test_bucket_assignment(orc):
    for eb, tensors, buckets in G.bucket_cases():
        bot, be = orc.assign_buckets(tensors, eb)
        assert list(be) == buckets, (eb, tensors)
        # every tensor lands in a bucket, in list order, contiguously
        assert list(bot) == sorted(bot)
        for b, size in enumerate(buckets):
            assert sum(t for t, k in zip(tensors, bot) if k == b) == size
    bot, be = orc.assign_buckets([], 4)
    assert len(be) == 0
