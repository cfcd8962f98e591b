"""Hierarchical (topology-aware) order on the GPU against the oracle, bit for bit: nodes of L
consecutive ranks, a ring inside each node over the segments of torch.chunk(chunk, L), then the
node sums by the tree rule.  Both paths that take the order are covered: gq_quantize +
gq_reduce_dequant, and the pipelined fused kernel; the other fused calls must refuse it."""
import numpy as np
import pytest
import torch

import dp_gradient_bucket_gb300 as gq
import oracle
import workloads as wl
import _gpu as H

pytestmark = pytest.mark.gpu

# (W, L): node sizes from one-rank nodes (the tree order) to one node (the ring order), odd node
# sizes and node counts (an odd node sum carried up a level), and the largest group
SHAPES = [(8, 2), (8, 4), (8, 8), (8, 1), (16, 4), (64, 8), (6, 3), (12, 4), (12, 3), (3, 3), (5, 1), (4, 2),
          (24, 8)]


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


def _host(cfg, W, n):
    stride = gq.row_stride(max(n, 1), 4)
    host = np.zeros(W * stride, dtype=np.float32)
    for r in range(W):
        wl.fill(cfg, r, 0, n, host[r * stride:r * stride + n])
    return host, stride


@pytest.mark.parametrize("W,L", SHAPES)
@pytest.mark.parametrize("mode", ["two_kernel", "pipe"])
def test_hier_ragged_buckets(W, L, mode):
    """Odd bucket sizes (chunks off the 16-byte grid, node segments of every length), an empty
    bucket, buckets shorter than L, and a chunk larger than the pipelined kernel's ring."""
    buckets = [5, 0, 1, 65535, 131075, 7, 32769 * 3 + 1, 3, 49152]
    n = sum(buckets)
    host, stride = _host(2, W, n)
    out, codes, scales, off, st = H.run(host, W, stride, buckets, "hier%d" % L, mode=mode)
    assert st == gq.GQ_OK
    H.compare_full(host, W, stride, off, oracle.HIER(L), 1.0, out, codes, scales)


@pytest.mark.parametrize("mode", ["two_kernel", "pipe"])
def test_hier_headline_bucket(mode):
    """The 25 MiB fp32 bucket at W = 8 in two nodes of four ranks, whole output."""
    W, n = 8, 6553600
    host, stride = wl.rows(2, W, n)
    out, codes, scales, off, st = H.run(host, W, stride, [n], "hier4", mode=mode)
    assert st == gq.GQ_OK and len(off) == 201
    H.compare_full(host, W, stride, off, oracle.HIER(4), 1.0, out, codes, scales)


@pytest.mark.parametrize("L", [1, 2, 8])
def test_hier_limits_match_ring_and_tree(L):
    """L = W is the ring order and L = 1, 2 the tree order: the GPU results agree bit for bit."""
    W, n = 8, 3 * 32768 + 4099
    host, stride = _host(1, W, n)
    hier = H.run(host, W, stride, [n], "hier%d" % L, mode="pipe")[0]
    other = H.run(host, W, stride, [n], "ring" if L == W else "tree", mode="pipe")[0]
    H.assert_bits_equal(hier[:n], other[:n], "hier%d against %s" % (L, "ring" if L == W else "tree"))


def test_hier_fp16_unscale():
    """fp16 gradients with a loss scale of 65536, W = 16 in four nodes."""
    W, L = 16, 4
    n = 65536 * 3 + 1001
    stride = gq.row_stride(n, 2)
    rng = np.random.default_rng(41)
    g = (rng.standard_normal((W, n)) * 1e-3 * 65536.0).astype(np.float16)
    host = np.zeros(W * stride, dtype=np.float16)
    for r in range(W):
        host[r * stride:r * stride + n] = g[r]
    for mode in ("two_kernel", "pipe"):
        out, codes, scales, off, st = H.run(host, W, stride, [n], "hier%d" % L, loss_scale=65536.0, mode=mode)
        assert st == gq.GQ_OK
        H.compare_full(host, W, stride, off, oracle.HIER(L), 65536.0, out, codes, scales)


def test_hier_refused_by_other_fused_calls():
    W, n = 8, 4096
    host, stride = _host(1, W, n)
    dev = torch.device("cuda:0")
    grads = torch.from_numpy(host).to(dev)
    nc, d_off = H.plan_device([n], 4, dev)
    out = torch.zeros(stride, dtype=torch.float32, device=dev)
    ws = torch.zeros(gq.gq_fused_workspace_bytes(nc, W) // 4, dtype=torch.int32, device=dev)
    order = gq.GQ_ORDER_HIER_NODES(4)
    with pytest.raises(gq.GQError) as e:
        gq.gq_fused_allreduce_sim(grads, W, stride, d_off, nc, 1.0, order, out)
    assert e.value.status == gq.GQ_ERR_UNSUPPORTED
    with pytest.raises(gq.GQError) as e:
        gq.gq_fused_allreduce_sim_ws(grads, W, stride, d_off, nc, 1.0, order, out, ws)
    assert e.value.status == gq.GQ_ERR_UNSUPPORTED
    assert gq.gq_get_error() == gq.GQ_OK
