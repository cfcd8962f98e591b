"""The adaptive chunk-size chooser (host logic) on a synthetic latency model."""
import numpy as np
import pytest

import __graft_entry__

__graft_entry__.build()  # the package loads libgq.so on import (it has no fallback)
from dp_gradient_bucket_gb300.chunker import DynamicChunker


def _latency(chunk, nbytes, rng, best=256 * 1024):
    # per-byte cost with a minimum at `best` (fixed per-chunk overhead against a tail that grows
    # with the chunk), plus 5% noise
    per_chunk_overhead = 2e-6
    chunks = max(1, nbytes // chunk)
    t = nbytes / 3.0e12 + chunks * per_chunk_overhead / 152 + (chunk / best) ** 2 * 4e-6
    return t * (1.0 + 0.05 * rng.standard_normal())


def test_measures_every_candidate_first_then_converges():
    rng = np.random.default_rng(1)
    ch = DynamicChunker(explore_every=0)
    nbytes = 209715200
    seen = []
    for _ in range(200):
        c = ch.predict_optimal()
        seen.append(c)
        ch.update_metrics(c, _latency(c, nbytes, rng), nbytes)
    assert seen[:len(ch.candidates)] == ch.candidates
    model = {c: _latency(c, nbytes, np.random.default_rng(0)) for c in ch.candidates}
    true_best = min(model, key=model.get)
    assert ch.best() == true_best
    assert seen[-50:].count(true_best) >= 45


def test_reexplores_the_stalest_candidate():
    ch = DynamicChunker(candidates=(1, 2, 3), explore_every=4)
    for c, lat in ((1, 3.0), (2, 1.0), (3, 2.0)):
        assert ch.predict_optimal() == c
        ch.update_metrics(c, lat, 1)
    picks = []
    for _ in range(8):
        c = ch.predict_optimal()
        picks.append(c)
        ch.update_metrics(c, {1: 3.0, 2: 1.0, 3: 2.0}[c], 1)
    # calls 4 and 8 re-measure the candidate measured longest ago (1, then 3); the rest exploit 2
    assert picks == [1, 2, 2, 2, 3, 2, 2, 2]


def test_ewma_and_bounded_history():
    ch = DynamicChunker(candidates=(10,), alpha=0.5, history=3)
    for lat in (4.0, 2.0, 2.0, 8.0):
        ch.update_metrics(10, lat, 2)
    # e = 2; 0.5 * 1 + 0.5 * 2 = 1.5; 1.25; 0.5 * 4 + 0.5 * 1.25 = 2.625
    assert ch.ewma[10] == pytest.approx(2.625)
    assert list(ch.history) == [(10, 2.0), (10, 2.0), (10, 8.0)]


def test_rejects_bad_input():
    with pytest.raises(ValueError):
        DynamicChunker(candidates=())
    with pytest.raises(ValueError):
        DynamicChunker(alpha=0.0)
    ch = DynamicChunker(candidates=(64,))
    with pytest.raises(ValueError):
        ch.update_metrics(65, 1.0, 1)
    with pytest.raises(ValueError):
        ch.update_metrics(64, 0.0, 1)
