"""The oracle against an exact-rational restatement (tests/_exact.py) on small seeded
inputs: every division, product, sum and the mean are re-derived in Fractions with an
explicit round-to-nearest-even to binary32, so a wrong operand, sign, index, order or
rounding rule in the oracle's float code shows up here."""
from fractions import Fraction

import numpy as np
import pytest

import _exact as X


def _values(rng, n, kind):
    if n == 0:
        return np.zeros(0, dtype=np.float32)
    if kind == "normal":
        return (rng.standard_normal(n) * 1e-3).astype(np.float32)
    if kind == "laplace_zeros":
        v = rng.laplace(0, 1e-4, n)
        v[rng.random(n) < 0.3] = 0.0
        out = rng.random(n) < 0.05
        v[out] *= 100
        return v.astype(np.float32)
    if kind == "subnormal":
        k = rng.integers(-300, 300, n)
        return (k.astype(np.float64) * 2.0 ** -149).astype(np.float32)
    if kind == "ties":
        e = int(rng.integers(-30, 10))
        k = rng.integers(-127, 127, n).astype(np.float64) + 0.5
        v = (k * 2.0 ** e).astype(np.float32)
        v[int(rng.integers(0, n))] = np.float32(127 * 2.0 ** e) * (1 if rng.random() < 0.5 else -1)
        return v
    if kind == "wide":
        return (rng.standard_normal(n) * 10.0 ** rng.uniform(-30, 30, n)).astype(np.float32)
    raise ValueError(kind)


KINDS = ["normal", "laplace_zeros", "subnormal", "ties", "wide"]


def _case(seed, W, kind):
    rng = np.random.default_rng(seed)
    # ragged chunk table: lengths 0..23, some shorter than W
    lens = rng.integers(0, 24, int(rng.integers(1, 6)))
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    n = int(off[-1])
    stride = n + int(rng.integers(0, 5))
    grads = np.zeros(W * stride, dtype=np.float32)
    for r in range(W):
        for j in range(len(lens)):
            lo, hi = off[j], off[j + 1]
            k = kind if kind != "mixed" else KINDS[int(rng.integers(0, len(KINDS)))]
            grads[r * stride + lo:r * stride + hi] = _values(rng, hi - lo, k)
    return grads, stride, off


@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 6, 8, 12])
@pytest.mark.parametrize("kind", KINDS + ["mixed"])
def test_quantize_reduce_exact(orc, W, kind):
    for seed in range(3):
        grads, stride, off = _case(1000 * W + 17 * seed + len(kind), W, kind)
        codes, scales, nf = orc.quantize(grads, W, stride, off)
        assert nf == 0
        nc = len(off) - 1
        for r in range(W):
            for j in range(nc):
                lo, hi = int(off[j]), int(off[j + 1])
                g = grads[r * stride + lo:r * stride + hi]
                q, s = X.quantize_chunk(g)
                assert X.bits(scales[r, j]) == X.bits(s), (r, j)
                assert list(codes[r * stride + lo:r * stride + hi]) == q, (r, j)
        for order in (orc.SEQ, orc.RING, orc.TREE):
            out = orc.reduce(codes, scales, W, stride, off, order)
            for j in range(nc):
                lo, hi = int(off[j]), int(off[j + 1])
                for i in range(lo, hi):
                    t = X.segment_of(i, lo, hi, W)
                    qs = [codes[r * stride + i] for r in range(W)]
                    ss = [scales[r, j] for r in range(W)]
                    want = X.reduce_element(qs, ss, order, t)
                    assert X.bits(out[i]) == X.bits(want), (order, j, i)
        for L in [L for L in range(1, W + 1) if W % L == 0]:
            out = orc.reduce(codes, scales, W, stride, off, orc.HIER(L))
            for j in range(nc):
                lo, hi = int(off[j]), int(off[j + 1])
                for i in range(lo, hi):
                    t = X.segment_of(i, lo, hi, L)
                    qs = [codes[r * stride + i] for r in range(W)]
                    ss = [scales[r, j] for r in range(W)]
                    want = X.reduce_element_hier(qs, ss, L, t)
                    assert X.bits(out[i]) == X.bits(want), (L, j, i)


@pytest.mark.parametrize("loss_scale", [65536.0, 1024.0, 3.0, 1.0])
def test_f16_unscale_exact(orc, loss_scale):
    rng = np.random.default_rng(int(loss_scale))
    W, n = 3, 40
    bits = rng.integers(0, 1 << 16, W * n).astype(np.uint16)
    bits[(bits & 0x7C00) == 0x7C00] = 0x3C00  # no inf / nan
    h = bits.view(np.float16)
    off = np.array([0, 13, 13, 40], dtype=np.int64)
    codes, scales, nf = orc.quantize(h, W, n, off, loss_scale=loss_scale)
    assert nf == 0
    inv = np.float32(1.0 / loss_scale)  # (float)(1.0 / (double)loss_scale)
    for r in range(W):
        for j in range(3):
            lo, hi = off[j], off[j + 1]
            g = [X.rn32(X.frac(np.float32(x)) * X.frac(inv)) for x in h[r * n + lo:r * n + hi]]
            q, s = X.quantize_chunk(g)
            assert X.bits(scales[r, j]) == X.bits(s)
            assert list(codes[r * n + lo:r * n + hi]) == q


def test_half_decode_all_patterns(orc):
    """Every binary16 pattern decodes to the value numpy's float16 -> float32 gives."""
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = allbits.view(np.float16).astype(np.float32)
    got = np.array([orc.half_to_float(b) for b in allbits], dtype=np.float32)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_mean_division_nonpower_of_two(orc):
    """out = acc / W is a correctly rounded division for W = 3, 5, 6, 7."""
    for W in (3, 5, 6, 7):
        rng = np.random.default_rng(W)
        n = 64
        grads = rng.standard_normal(W * n).astype(np.float32)
        off = np.array([0, n], dtype=np.int64)
        codes, scales, _ = orc.quantize(grads, W, n, off)
        out = orc.reduce(codes, scales, W, n, off, orc.SEQ)
        for i in range(n):
            d = [X.rn32(Fraction(int(codes[r * n + i])) * X.frac(scales[r, 0])) for r in range(W)]
            acc = X.sum_in_order(d)
            assert X.bits(out[i]) == X.bits(X.rn32(X.frac(acc) / W))
