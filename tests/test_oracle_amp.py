"""Pins of the oracle's mixed-precision pieces: the loss-scale update (hand-derived sequence, the
overflow guard, closed forms) and the non-finite count that drives the found-inf flag (brute force)."""
import numpy as np

import oracle
import workloads as wl

GOLDEN = __file__.replace("test_oracle_amp.py", "golden/amp_update.txt")


def test_update_sequence_golden():
    scale, tracker = np.float32(65536.0), 0
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    assert len(rows) == 13
    for f, want_scale, want_tracker in rows:
        scale, tracker = oracle.amp_update_scale(scale, tracker, float(f), 2.0, 0.5, 3)
        assert scale == np.float32(float(want_scale)) and tracker == int(want_tracker), (f, scale, tracker)


def test_growth_that_overflows_keeps_the_scale():
    big = np.float32(2.0 ** 127)
    scale, tracker = oracle.amp_update_scale(big, 0, 0.0, 2.0, 0.5, 1)
    assert scale == big and tracker == 0
    scale, tracker = oracle.amp_update_scale(big, 4, 0.0, 2.0, 0.5, 5)
    assert scale == big and tracker == 0


def test_backoff_rounds_like_binary32():
    # 3 * 0.1f rounds to the binary32 nearest the exact product of the two binary32 values
    s, _ = oracle.amp_update_scale(np.float32(3.0), 7, 1.0, 2.0, np.float32(0.1), 100)
    exact = 3 * float(np.float32(0.1))
    assert s == np.float32(exact)


def test_closed_form_over_long_runs():
    """With power-of-two factors no rounding happens: after any sequence, log2(scale) moves by +1
    per completed run of `interval` clean steps (never past 127, where growth would overflow) and
    -1 per overflow."""
    rng = np.random.default_rng(5)
    for interval in (1, 2, 7, 2000):
        scale, tracker = np.float32(2.0 ** 16), 0
        expect_log, run = 16, 0
        for f in rng.random(6000) < 0.01:
            scale, tracker = oracle.amp_update_scale(scale, tracker, float(f), 2.0, 0.5, interval)
            if f:
                expect_log, run = expect_log - 1, 0
            else:
                run += 1
                if run == interval:
                    expect_log, run = min(expect_log + 1, 127), 0
            assert scale == np.float32(2.0 ** expect_log) and tracker == run


def test_nonfinite_count_brute_force():
    """The count of (rank, chunk) pairs holding an Inf or NaN, or a value that overflows when unscaled."""
    W, n = 3, 70001
    stride = 70004
    host = np.zeros(W * stride, dtype=np.float32)
    for r in range(W):
        wl.fill(1, r, 0, n, host[r * stride:r * stride + n])
    off = oracle.plan_chunks([n], 4)
    assert len(off) - 1 == 2
    host[0 * stride + 3] = np.inf
    host[0 * stride + 10] = np.nan          # same (rank, chunk): counted once
    host[2 * stride + 60000] = -np.inf
    _, _, nf = oracle.quantize(host, W, stride, off)
    assert nf == 2
    # a finite value that overflows once unscaled by a loss scale below one
    h2 = np.zeros(W * stride, dtype=np.float32)
    h2[1 * stride + 5] = np.float32(3e38)
    _, _, nf = oracle.quantize(h2, W, stride, off, loss_scale=0.5)
    assert nf == 1
    _, _, nf = oracle.quantize(h2, W, stride, off, loss_scale=1.0)
    assert nf == 0
