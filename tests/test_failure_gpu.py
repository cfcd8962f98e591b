"""Failure detection without a GPU fault: a device-side wait that cannot complete gives up
after its limit, the kernel records GQ_ERR_TIMEOUT and returns, and the context stays
usable (the next call is bit-exact).  The stall is injected from the host: the bulk-copy
barrier is told to expect 16 bytes more than the copies deliver."""
import numpy as np
import pytest
import torch

import dp_gradient_bucket_gb300 as gq
import oracle
import workloads as wl
import _gpu as H

pytestmark = pytest.mark.gpu


def test_bulk_copy_wait_runs_out_and_is_reported():
    # W = 4 runs the cluster kernel that stages each slice in shared memory with bulk copies (the
    # W = 8 register-staged kernel has no bulk-copy wait); 8 chunks of 32,768
    W, n = 4, 262144
    host, stride = wl.rows(2, W, n)
    off = oracle.plan_chunks([n], 4)
    assert gq.gq_get_error() == gq.GQ_OK
    try:
        gq.gq_testing_inject_copy_stall(16, 2_000_000)   # 2 ms limit
        _, _, _, _, st = H.run(host, W, stride, [n], "ring", want_codes=False)
        assert st == gq.GQ_ERR_TIMEOUT
    finally:
        gq.gq_testing_inject_copy_stall(0, 0)
    out, codes, scales, _, st = H.run(host, W, stride, [n], "ring")
    assert st == gq.GQ_OK
    H.compare_full(host, W, stride, off, oracle.RING, 1.0, out, codes, scales)
    torch.cuda.synchronize()
