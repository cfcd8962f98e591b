"""Scale scopes and the base chunk size on the GPU against the oracle, bit for bit: one scale per
tensor or per bucket (gq_plan_chunks_ex with GQ_SCOPE_TENSOR / GQ_SCOPE_BUCKET), and dynamic_chunk
with other base chunk sizes (the CHUNK_SIZE knob), through the two-kernel path and the pipelined
kernel.  The device table is compared with the oracle's too."""
import numpy as np
import pytest
import torch

import dp_gradient_bucket_gb300 as gq
import oracle
import workloads as wl
import _gpu as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


@pytest.fixture(scope="module")
def resnet_rows():
    """The ResNet-152-sized gradient layout (workload 3), W = 8: its tensor sizes and buckets."""
    sizes, _ = wl.tensor_layout(3)
    n = int(sizes.sum())
    host, stride = wl.rows(3, 8, n)
    buckets = oracle.assign_buckets([int(x) for x in sizes], 4)[1]
    return host, stride, [int(x) for x in sizes], [int(x) for x in buckets]


@pytest.mark.parametrize("mode", ["pipe", "two_kernel"])
def test_per_tensor_scale_resnet_layout(resnet_rows, mode):
    """One scale per tensor (about 270 tensors of 64 to 2.36 M elements, the largest read twice
    by the pipelined kernel), ring segments per tensor, whole output."""
    host, stride, sizes, _ = resnet_rows
    W = 8
    out, codes, scales, off, st = H.run(host, W, stride, sizes, "ring", mode=mode, scope="tensor")
    assert st == gq.GQ_OK
    assert np.array_equal(off, oracle.plan_chunks_ex(sizes, 4, oracle.SCOPE_TENSOR))
    H.compare_full(host, W, stride, off, oracle.RING, 1.0, out, codes, scales)


@pytest.mark.parametrize("mode", ["pipe", "two_kernel"])
def test_per_bucket_scale_resnet_layout(resnet_rows, mode):
    """One scale per 25 MiB bucket (about 10 chunks of up to 6.5 M elements), seq order."""
    host, stride, _, buckets = resnet_rows
    W = 8
    out, codes, scales, off, st = H.run(host, W, stride, buckets, "seq", mode=mode, scope="bucket")
    assert st == gq.GQ_OK
    assert np.array_equal(off, oracle.plan_chunks_ex(buckets, 4, oracle.SCOPE_BUCKET))
    H.compare_full(host, W, stride, off, oracle.SEQ, 1.0, out, codes, scales)


@pytest.mark.parametrize("chunk_bytes", [16384, 32868, 65536, 262144, 1 << 20])
def test_chunk_size_headline_bucket(chunk_bytes):
    """The 25 MiB fp32 bucket at W = 8 cut with other base chunk sizes (32868 is not a multiple
    of the 64-byte alignment), pipelined kernel, ring order, whole output."""
    W, n = 8, 6553600
    host, stride = wl.rows(2, W, n)
    out, codes, scales, off, st = H.run(host, W, stride, [n], "ring", mode="pipe", chunk_bytes=chunk_bytes)
    assert st == gq.GQ_OK
    assert np.array_equal(off, oracle.plan_chunks_ex([n], 4, oracle.SCOPE_CHUNK, chunk_bytes))
    H.compare_full(host, W, stride, off, oracle.RING, 1.0, out, codes, scales)


def test_per_tensor_scale_fp16_unscale():
    """fp16 gradients of twelve BERT-Large tensors after the embedding (workload 4 layout), W = 16,
    loss scale 65536, one scale per tensor, both paths."""
    sizes, _ = wl.tensor_layout(4)
    sizes = [int(x) for x in sizes[1:13]]
    n = sum(sizes)
    W = 16
    host, stride = wl.rows(4, W, n)
    for mode in ("pipe", "two_kernel"):
        out, codes, scales, off, st = H.run(host, W, stride, sizes, "ring", loss_scale=65536.0, mode=mode,
                                            scope="tensor")
        assert st == gq.GQ_OK
        H.compare_full(host, W, stride, off, oracle.RING, 65536.0, out, codes, scales)
