"""Exact-rational restatement of the quantise/reduce steps, used to pin the oracle.

Every value is a fractions.Fraction; each binary32 rounding is done explicitly by
`rn32` (nearest float32 by exact distance, ties to the even bit pattern), so nothing
here relies on the host's float division, rounding mode or contraction.  Slow: for
inputs of a few hundred elements.
"""
from fractions import Fraction

import numpy as np

F32_INF = np.float32(np.inf)


def frac(x):
    return Fraction(float(x))


def rn32(x):
    """Round the exact rational x to the nearest binary32 value, ties to even."""
    if x == 0:
        return np.float32(0.0)
    f = np.float32(float(x))  # within one ulp of the answer (double rounding may miss)
    cands = [f, np.nextafter(f, F32_INF), np.nextafter(f, -F32_INF)]
    cands = [c for c in cands if np.isfinite(c)]

    def key(c):
        return (abs(frac(c) - x), int(np.array(c, dtype=np.float32).view(np.uint32)) & 1)

    return min(cands, key=key)


def rint_even(y):
    """Nearest integer to the rational y, ties to even."""
    fl = y.numerator // y.denominator
    rem = y - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def quantize_chunk(g):
    """Codes and scale of one chunk: s = RN(max|g| / 127); q = clamp(rne(RN(g / s)))."""
    g = [np.float32(v) for v in g]
    m = max([abs(frac(v)) for v in g], default=Fraction(0))
    s = rn32(m / 127)
    if s == 0:
        return [0] * len(g), s
    codes = []
    for v in g:
        y = rn32(frac(v) / frac(s))
        q = rint_even(frac(y))
        codes.append(max(-128, min(127, q)))
    return codes, s


def segment_of(i, lo, hi, W):
    """Index of element i's piece in torch.chunk(chunk[lo:hi], W)."""
    seg = -(-(hi - lo) // W)
    return (i - lo) // seg


def rank_order(order, W, t):
    if order == 0:
        return list(range(W))
    if order == 1:
        return [(t + k) % W for k in range(1, W + 1)]
    raise ValueError(order)


def sum_in_order(terms):
    acc = terms[0]
    for d in terms[1:]:
        acc = rn32(frac(acc) + frac(d))
    return acc


def sum_tree(terms):
    level = list(terms)
    while len(level) > 1:
        nxt = [rn32(frac(level[p]) + frac(level[p + 1])) for p in range(0, len(level) - 1, 2)]
        if len(level) % 2:
            nxt.append(level[-1])
        level = nxt
    return level[0]


def reduce_element(qs, ss, order, t):
    """Mean over ranks of the dequantised values, summed in the given order."""
    W = len(qs)
    d = [rn32(Fraction(int(q)) * frac(s)) for q, s in zip(qs, ss)]
    if order == 2:
        acc = sum_tree(d)
    else:
        acc = sum_in_order([d[r] for r in rank_order(order, W, t)])
    return rn32(frac(acc) / W)


def reduce_element_hier(qs, ss, L, t):
    """Mean over ranks in the hierarchical order: nodes of L consecutive ranks, each summed in
    ring order from local rank (t+1) % L (t = segment in torch.chunk(chunk, L)), then the node
    sums pairwise in node order, an odd one carried."""
    W = len(qs)
    d = [rn32(Fraction(int(q)) * frac(s)) for q, s in zip(qs, ss)]
    nodes = [sum_in_order([d[n * L + (t + k) % L] for k in range(1, L + 1)]) for n in range(W // L)]
    return rn32(frac(sum_tree(nodes)) / W)


def bits(x):
    return int(np.array(x, dtype=np.float32).view(np.uint32))
