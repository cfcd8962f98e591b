"""Adaptive base chunk size for dynamic_chunk.

The "pipelined HCCL AllReduce" article (§6.2, adaptive chunking) sketches a DynamicChunker that
keeps a bounded history (100 entries) of (chunk size, latency) pairs and predicts the best chunk
size with an exponentially weighted moving average; the prediction's body is not given.  This
module specifies it:

  - candidates: a fixed list of base chunk sizes in bytes (the CHUNK_SIZE knob of §4.2, which
    gq_plan_chunks_ex takes as `chunk_bytes`);
  - update_metrics(chunk_size, latency, nbytes): appends to the bounded history and folds the
    latency per byte moved into that candidate's EWMA, e <- alpha * x + (1 - alpha) * e (the first
    sample sets e = x);
  - predict_optimal(): a candidate never measured comes first (in list order); otherwise, every
    `explore_every`-th call re-measures the candidate measured longest ago (the best size can move
    as the load changes); otherwise the candidate with the lowest EWMA (ties: the earlier one).

Host logic only: the latencies come from the caller (CUDA events around the call it times).
"""
from collections import deque

DEFAULT_CANDIDATES = (32 * 1024, 64 * 1024, 128 * 1024, 256 * 1024, 512 * 1024, 1024 * 1024)


class DynamicChunker:
    def __init__(self, candidates=DEFAULT_CANDIDATES, alpha=0.3, history=100, explore_every=50):
        if not candidates:
            raise ValueError("no candidate chunk sizes")
        if not 0.0 < alpha <= 1.0:
            raise ValueError("alpha must lie in (0, 1]")
        self.candidates = [int(c) for c in candidates]
        self.alpha = float(alpha)
        self.explore_every = int(explore_every)
        self.history = deque(maxlen=int(history))
        self.ewma = {}        # candidate -> EWMA of seconds per byte
        self.last_seen = {}   # candidate -> update count when last measured
        self.updates = 0
        self.calls = 0

    def update_metrics(self, chunk_size, latency, nbytes):
        chunk_size = int(chunk_size)
        if chunk_size not in self.candidates:
            raise ValueError("%d is not a candidate chunk size" % chunk_size)
        if not latency > 0 or not nbytes > 0:
            raise ValueError("latency and nbytes must be positive")
        self.history.append((chunk_size, float(latency)))
        x = float(latency) / float(nbytes)
        e = self.ewma.get(chunk_size)
        self.ewma[chunk_size] = x if e is None else self.alpha * x + (1.0 - self.alpha) * e
        self.updates += 1
        self.last_seen[chunk_size] = self.updates

    def predict_optimal(self):
        self.calls += 1
        for c in self.candidates:
            if c not in self.ewma:
                return c
        if self.explore_every > 0 and self.calls % self.explore_every == 0:
            return min(self.candidates, key=lambda c: (self.last_seen[c], self.candidates.index(c)))
        return min(self.candidates, key=lambda c: (self.ewma[c], self.candidates.index(c)))

    def best(self):
        """The candidate with the lowest EWMA so far (None before any measurement)."""
        if not self.ewma:
            return None
        return min(self.ewma, key=lambda c: (self.ewma[c], self.candidates.index(c)))
