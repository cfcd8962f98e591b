"""Invariants that the pages and the mathematics fix, checked on larger seeded inputs
(numpy, float64 checks), plus the all-ranks-equal self-test pattern."""
import numpy as np
import pytest

FLT_MIN = np.float32(2.0 ** -126)


def _grads(seed, W, n, kind="normal"):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return (rng.standard_normal(W * n) * 1e-3).astype(np.float32)
    v = rng.laplace(0, 1e-4, W * n)
    v[rng.random(W * n) < 0.3] = 0
    v[rng.random(W * n) < 0.001] *= 100
    return v.astype(np.float32)


@pytest.mark.parametrize("kind", ["normal", "laplace"])
def test_code_and_scale_invariants(orc, kind):
    W, n = 4, 200003
    grads = _grads(7, W, n, kind)
    off = orc.plan_chunks([n], 4)
    codes, scales, nf = orc.quantize(grads, W, n, off)
    assert nf == 0
    g = grads.reshape(W, n).astype(np.float64)
    q = codes.reshape(W, n).astype(np.float64)
    for r in range(W):
        for j in range(len(off) - 1):
            lo, hi = off[j], off[j + 1]
            s = np.float64(scales[r, j])
            m = np.abs(g[r, lo:hi]).max()
            assert s >= FLT_MIN
            # scale * 127 recovers max|g| within one ulp of m
            assert abs(s * 127 - m) <= np.spacing(np.float32(m))
            # codes within [-127, 127]; the largest magnitude maps to +-127
            assert q[r, lo:hi].min() >= -127 and q[r, lo:hi].max() <= 127
            i = lo + int(np.argmax(np.abs(g[r, lo:hi])))
            assert abs(q[r, i]) == 127
            # |dequant - g| <= s/2 (the fp32 quotient's rounding adds < 2^-22 relative)
            err = np.abs(q[r, lo:hi] * s - g[r, lo:hi])
            assert err.max() <= s / 2 * (1 + 2.0 ** -22)


def test_constant_ranks_self_test(orc):
    """Rank r holds the constant r + 1 (the all_reduce-of-ones*rank self-test pattern of the
    3D-parallel article): every code is 127 and the mean is (W + 1) / 2 within a few ulp."""
    for W in (1, 2, 3, 4, 8, 16):
        n = 4096 + 3
        grads = np.concatenate([np.full(n, r + 1, dtype=np.float32) for r in range(W)])
        off = orc.plan_chunks([n], 4)
        for order in (orc.SEQ, orc.RING, orc.TREE):
            out, codes, scales, _ = orc.fused(grads, W, n, off, order)
            assert np.all(codes == 127)
            want = (W + 1) / 2
            assert np.all(np.abs(out.astype(np.float64) - want) <= 4 * np.spacing(np.float32(want)))


def test_single_rank_is_dequant(orc):
    n = 70001
    grads = _grads(11, 1, n)
    off = orc.plan_chunks([n], 4)
    for order in (orc.SEQ, orc.RING, orc.TREE):
        out, codes, scales, _ = orc.fused(grads, 1, n, off, order)
        chunk = np.repeat(np.arange(len(off) - 1), np.diff(off))
        deq = (codes.astype(np.float32) * scales[0, chunk]).astype(np.float32)
        assert np.array_equal(out.view(np.uint32), deq.view(np.uint32))


def test_two_ranks_orders_agree(orc):
    """With W = 2 every order adds the same two terms: seq, ring and tree are identical."""
    n = 65537
    grads = _grads(13, 2, n, "laplace")
    off = orc.plan_chunks([n], 4)
    outs = [orc.fused(grads, 2, n, off, o)[0] for o in (orc.SEQ, orc.RING, orc.TREE)]
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    assert np.array_equal(outs[0].view(np.uint32), outs[2].view(np.uint32))


def test_hier_reduces_to_ring_and_tree(orc):
    """Hierarchical order: one node of W ranks is the ring order, W one-rank nodes the tree
    order, and nodes of two ranks the tree order too (a two-term sum does not depend on which
    term comes first, and the node sums are the tree's first level)."""
    for W in (2, 4, 6, 8, 12, 16):
        n = 3 * 32768 + 4099
        grads = _grads(17 + W, W, n, "laplace")
        off = orc.plan_chunks([n], 4)
        codes, scales, _ = orc.quantize(grads, W, n, off)
        ring = orc.reduce(codes, scales, W, n, off, orc.RING).view(np.uint32)
        tree = orc.reduce(codes, scales, W, n, off, orc.TREE).view(np.uint32)
        assert np.array_equal(orc.reduce(codes, scales, W, n, off, orc.HIER(W)).view(np.uint32), ring)
        assert np.array_equal(orc.reduce(codes, scales, W, n, off, orc.HIER(1)).view(np.uint32), tree)
        assert np.array_equal(orc.reduce(codes, scales, W, n, off, orc.HIER(2)).view(np.uint32), tree)


def test_hier_node_swap(orc):
    """With two nodes the top level is one commutative add: swapping the nodes' data leaves
    every output bit unchanged."""
    W, L, n = 8, 4, 4 * 8192 + 5
    grads = _grads(29, W, n, "laplace").reshape(W, n)
    off = orc.plan_chunks([n], 4)
    out = orc.fused(grads.reshape(-1), W, n, off, orc.HIER(L))[0]
    swapped = np.concatenate([grads[L:], grads[:L]])
    out2 = orc.fused(swapped.reshape(-1), W, n, off, orc.HIER(L))[0]
    assert np.array_equal(out.view(np.uint32), out2.view(np.uint32))


def test_hier_node_rotation_shifts_segments(orc):
    """Node ring schedule: segment t starts at local rank (t+1) % L.  With every row constant,
    rotating each node's ranks by one (new local k holds old local k+1) makes segment t add the
    same terms in the order that segment t+1 used before, so the per-segment results shift by
    one segment, bit for bit."""
    W, L, n = 8, 4, 4 * 8192
    rng = np.random.default_rng(29)
    consts = (rng.standard_normal(W) * 10.0 ** rng.uniform(-4, 4, W)).astype(np.float32)
    rows = np.repeat(consts[:, None], n, axis=1)
    off = np.array([0, n], dtype=np.int64)
    seg = n // L
    a = orc.fused(rows.reshape(-1), W, n, off, orc.HIER(L))[0].view(np.uint32)
    rot = np.concatenate([np.roll(rows[b * L:(b + 1) * L], -1, axis=0) for b in range(W // L)])
    b = orc.fused(rot.reshape(-1), W, n, off, orc.HIER(L))[0].view(np.uint32)
    per_seg = [a[t * seg] for t in range(L)]
    assert len(set(per_seg)) > 1  # the orders really round differently on this data
    for t in range(L):
        assert np.all(a[t * seg:(t + 1) * seg] == per_seg[t])
        assert np.all(b[t * seg:(t + 1) * seg] == per_seg[(t + 1) % L]), t


def test_hier_rejects_nondividing_node_size(orc):
    grads = _grads(3, 6, 100)
    off = np.array([0, 100], dtype=np.int64)
    codes, scales, _ = orc.quantize(grads, 6, 100, off)
    with pytest.raises(ValueError):
        orc.reduce(codes, scales, 6, 100, off, orc.HIER(4))


def test_quantisation_error_against_unquantised_mean(orc):
    """Turning quantisation off changes the mean by at most (1/W) * sum_r s_r / 2 plus
    rounding of the W-term sum (the page's 'disable quantisation to check precision')."""
    W, n = 8, 131072
    grads = _grads(17, W, n, "laplace")
    off = orc.plan_chunks([n], 4)
    out, codes, scales, _ = orc.fused(grads, W, n, off, orc.RING)
    exact = grads.reshape(W, n).astype(np.float64).mean(axis=0)
    chunk = np.repeat(np.arange(len(off) - 1), np.diff(off))
    bound = scales[:, chunk].astype(np.float64).sum(axis=0) / (2 * W)
    slack = (np.abs(grads.reshape(W, n)).astype(np.float64).sum(axis=0) / W) * W * 2.0 ** -23 + 1e-45
    assert np.all(np.abs(out - exact) <= bound * (1 + 2.0 ** -20) + slack)


def test_tree_within_tolerance_of_seq(orc):
    W, n = 16, 100000
    grads = _grads(19, W, n, "laplace")
    off = orc.plan_chunks([n], 4)
    seq, codes, scales, _ = orc.fused(grads, W, n, off, orc.SEQ)
    tree = orc.reduce(codes, scales, W, n, off, orc.TREE)
    chunk = np.repeat(np.arange(len(off) - 1), np.diff(off))
    terms = np.abs(codes.reshape(W, n).astype(np.float64) * scales[:, chunk]).sum(axis=0) / W
    assert np.all(np.abs(tree.astype(np.float64) - seq) <= 1e-6 * terms + 1e-45)


def test_nonfinite_chunks_are_counted(orc):
    n = 1000
    grads = np.zeros(2 * n, dtype=np.float32)
    grads[5] = np.inf
    grads[n + 7] = np.nan
    codes, scales, nf = orc.quantize(grads, 2, n, np.array([0, 500, 1000]))
    assert nf == 2
