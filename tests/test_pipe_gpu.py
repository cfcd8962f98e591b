"""gq_fused_allreduce_sim_pipelined (the quantise / reduce pipeline through L2) against the oracle,
through the C ABI: the cases particular to it.  The common workloads and edge cases run it from
test_parity_gpu.py (mode "pipe")."""
import numpy as np
import pytest
import torch

import dp_gradient_bucket_gb300 as gq
import oracle
import workloads as wl
import _gpu as H

pytestmark = pytest.mark.gpu

ORDERS = [("seq", oracle.SEQ), ("ring", oracle.RING), ("tree", oracle.TREE)]


@pytest.fixture(scope="module", autouse=True)
def _device():
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


def _ws(W, stride, nc, dev):
    return torch.zeros(gq.gq_pipelined_workspace_bytes(W, stride, nc), dtype=torch.uint8, device=dev)


@pytest.mark.parametrize("W", [3, 8])
@pytest.mark.parametrize("order,oorder", ORDERS)
def test_pipe_chunks_larger_than_the_ring(W, order, oorder):
    """A hand-made table with chunks far longer than the shared-memory ring (copied once per
    pass), chunk starts off the 16-byte grid, a 3-element chunk and an empty one."""
    n = 460000
    stride = gq.row_stride(n, 4)
    host = np.zeros(W * stride, dtype=np.float32)
    for r in range(W):
        wl.fill(2, r, 0, n, host[r * stride:r * stride + n])
    table = np.array([0, 3, 200003, 200010, 450001, 450001, 460000], dtype=np.int64)
    out, codes, scales, _, st = H.run(host, W, stride, None, order, mode="pipe", offsets=table)
    assert st == gq.GQ_OK
    H.compare_full(host, W, stride, table, oorder, 1.0, out[:n], codes, scales)


@pytest.mark.parametrize("W,dt", [(64, np.float32), (48, np.float32), (64, np.float16)])
def test_pipe_many_items_per_cta_with_two_pass_chunks(W, dt):
    """Many rank-chunks per CTA, two-pass chunks (longer than the ring) between single-pass ones:
    a quantiser warp may reach a ring slot while the slot's previous piece is still in flight (bulk
    copies land in any order).  Each call on a fresh workspace, several calls."""
    eb = np.dtype(dt).itemsize
    big = (262144 - 4) // eb  # one chunk of 256 KiB less one element: copied once per pass
    buckets = [5, 0, 1, big, 131075 * 4 // eb, 7, big, 32769 * 3 + 1, 3, 196608 // eb, big]
    n = sum(buckets)
    stride = gq.row_stride(n, eb)
    host = np.zeros(W * stride, dtype=dt)
    for r in range(W):
        wl.fill(4 if dt == np.float16 else 2, r, 0, n, host[r * stride:r * stride + n])
    ls = 65536.0 if dt == np.float16 else 1.0
    want = None
    for rep in range(4):
        out, codes, scales, off, st = H.run(host, W, stride, buckets, "ring", loss_scale=ls, mode="pipe")
        assert st == gq.GQ_OK, "call %d" % rep
        if want is None:
            H.compare_full(host, W, stride, off, oracle.RING, ls, out, codes, scales)
            want = out.copy()
        else:
            H.assert_bits_equal(out, want, "output of call %d" % rep)


@pytest.mark.parametrize("max_ctas", [1, 7, 40, 100000])
def test_pipe_capped_grid(max_ctas):
    """The capped grid (gq_fused_allreduce_sim_pipelined_ex) gives the same bits for any cap, down to
    one CTA doing every item of both stages."""
    W, n = 8, 300007
    host, stride = wl.rows(2, W, n)
    dev = torch.device("cuda:0")
    grads = torch.from_numpy(host).to(dev)
    nc, d_off = H.plan_device([n], 4, dev)
    out = torch.zeros(n, dtype=torch.float32, device=dev)
    ws = _ws(W, stride, nc, dev)
    want = oracle.fused(host, W, stride, d_off.cpu().numpy(), oracle.RING)[0]
    for _ in range(2):
        gq.gq_fused_allreduce_sim_pipelined(grads, W, stride, d_off, nc, 1.0, "ring", out, ws, max_ctas=max_ctas)
        assert gq.gq_get_error() == gq.GQ_OK
        H.assert_bits_equal(out.cpu().numpy(), want, "output")
    assert H.pipe_header(ws) == (0, 0, 0, 2)


@pytest.mark.parametrize("W", [8, 16])
def test_pipe_fp16_unscale(W):
    """fp16 gradients with loss scales 65536 (exact unscale) and 3 (inexact), every order."""
    n = 300007
    stride = gq.row_stride(n, 2)
    host = np.zeros(W * stride, dtype=np.float16)
    for r in range(W):
        wl.fill(4, r, 0, n, host[r * stride:r * stride + n])
    for ls in (65536.0, 3.0):
        for order, oorder in ORDERS:
            out, codes, scales, off, st = H.run(host, W, stride, [n], order, loss_scale=ls, mode="pipe")
            assert st == gq.GQ_OK
            H.compare_full(host, W, stride, off, oorder, ls, out, codes, scales)


def test_pipe_many_calls_and_workspace_after_bad_table():
    """Ten calls in a row on one workspace give the same bits (the words of one call are never
    taken for the next one's, and the codes discarded from L2 by one call are rewritten by the
    next); after a call that reports a bad table the workspace still serves; a different table on
    the same workspace works too."""
    W, n = 8, 1 << 20
    host, stride = wl.rows(5, W, n)
    dev = torch.device("cuda:0")
    grads = torch.from_numpy(host).to(dev)
    nc, d_off = H.plan_device([n], 4, dev)
    want = oracle.fused(host, W, stride, d_off.cpu().numpy(), oracle.RING)[0]
    ws = _ws(W, stride, nc, dev)
    out = torch.empty(n, dtype=torch.float32, device=dev)

    def check():
        out.fill_(0)
        gq.gq_fused_allreduce_sim_pipelined(grads, W, stride, d_off, nc, 1.0, "ring", out, ws)
        assert gq.gq_get_error() == gq.GQ_OK
        H.assert_bits_equal(out.cpu().numpy(), want, "output")
        assert H.pipe_header(ws)[:3] == (0, 0, 0)

    for k in range(10):
        check()
        assert H.pipe_header(ws)[3] == k + 1  # one launch counted per call
    bad = torch.tensor([0, 1000, 5000, 2000, 3000], dtype=torch.int64, device=dev)
    gq.gq_fused_allreduce_sim_pipelined(grads, W, stride, bad, 4, 1.0, "ring", out, ws)
    assert gq.gq_get_error() == gq.GQ_ERR_BAD_TABLE
    check()
    small = np.array([0, 40000, 70001, 70001, 100003], dtype=np.int64)
    d_small = torch.from_numpy(small).to(dev)
    gq.gq_fused_allreduce_sim_pipelined(grads, W, stride, d_small, 4, 1.0, "seq", out, ws)
    assert gq.gq_get_error() == gq.GQ_OK
    s2 = gq.row_stride(100003, 4)
    rows = np.zeros((W, s2), dtype=np.float32)
    rows[:, :100003] = host.reshape(W, stride)[:, :100003]
    H.assert_bits_equal(out.cpu().numpy()[:100003], oracle.fused(rows.reshape(-1), W, s2, small, oracle.SEQ)[0],
                        "small table")
    check()


def test_pipe_epoch_wrap_clears_words():
    """A workspace whose launch counter is one short of wrapping: that call clears every word and
    restarts the counter, and the calls on either side of the wrap give the same bits."""
    W, n = 8, 300001
    host, stride = wl.rows(1, W, n)
    dev = torch.device("cuda:0")
    grads = torch.from_numpy(host).to(dev)
    nc, d_off = H.plan_device([n], 4, dev)
    want = oracle.fused(host, W, stride, d_off.cpu().numpy(), oracle.SEQ)[0]
    ws = _ws(W, stride, nc, dev)
    out = torch.empty(n, dtype=torch.float32, device=dev)
    gq.gq_fused_allreduce_sim_pipelined(grads, W, stride, d_off, nc, 1.0, "seq", out, ws)
    assert gq.gq_get_error() == gq.GQ_OK
    ws.view(torch.int32)[5] = -2  # launch counter 0xfffffffe: the next call tags its words 0xffffffff
    words = nc * W * 8
    for k in range(3):
        out.fill_(0)
        gq.gq_fused_allreduce_sim_pipelined(grads, W, stride, d_off, nc, 1.0, "seq", out, ws)
        assert gq.gq_get_error() == gq.GQ_OK
        H.assert_bits_equal(out.cpu().numpy(), want, "output %d" % k)
        if k == 0:
            assert H.pipe_header(ws)[3] == 0
            assert int(ws[256:256 + words].to(torch.int32).abs().sum().item()) == 0  # every word cleared
        else:
            assert H.pipe_header(ws)[3] == k


@pytest.mark.parametrize("W", [4, 8])
def test_pipe_found_inf_flag(W):
    """found_inf is set by an Inf, a NaN, or an fp16 value that overflows when unscaled, and left
    alone by clean data; the finite chunks still match the oracle."""
    dev = torch.device("cuda:0")
    n = 300000
    stride = gq.row_stride(n, 4)
    host = np.zeros(W * stride, dtype=np.float32)
    for r in range(W):
        wl.fill(1, r, 0, n, host[r * stride:r * stride + n])
    grads = torch.from_numpy(host).to(dev)
    nc, d_off = H.plan_device([n], 4, dev)
    ws = _ws(W, stride, nc, dev)
    out = torch.empty(n, dtype=torch.float32, device=dev)
    flag = torch.zeros(1, dtype=torch.float32, device=dev)
    gq.gq_fused_allreduce_sim_pipelined(grads, W, stride, d_off, nc, 1.0, "ring", out, ws, found_inf=flag)
    assert gq.gq_get_error() == gq.GQ_OK and float(flag.item()) == 0.0
    bad = host.copy()
    bad[1 * stride + 7] = np.nan
    gq.gq_fused_allreduce_sim_pipelined(torch.from_numpy(bad).to(dev), W, stride, d_off, nc, 1.0, "ring", out, ws,
                                        found_inf=flag)
    assert gq.gq_get_error() == gq.GQ_WARN_NONFINITE and float(flag.item()) == 1.0
    off = d_off.cpu().numpy()
    want = oracle.fused(host, W, stride, off, oracle.RING)[0]
    got = out.cpu().numpy()
    H.assert_bits_equal(got[off[1]:], want[off[1]:], "finite chunks")
    # fp16 with a loss scale below 1: 60000 * (1 / 1e-35) overflows binary32 when unscaled
    h = np.zeros(W * gq.row_stride(n, 2), dtype=np.float16)
    s2 = gq.row_stride(n, 2)
    h[3 * s2 + 11] = np.float16(60000.0)
    flag.zero_()
    nc2, d_off2 = H.plan_device([n], 2, dev)
    ws2 = _ws(W, s2, nc2, dev)
    gq.gq_fused_allreduce_sim_pipelined(torch.from_numpy(h).to(dev), W, s2, d_off2, nc2, 1e-35, "ring", out, ws2,
                                        found_inf=flag)
    assert gq.gq_get_error() == gq.GQ_WARN_NONFINITE and float(flag.item()) == 1.0


def test_pipe_non_default_stream():
    W, n = 8, 500001
    stride = gq.row_stride(n, 4)
    host = np.zeros(W * stride, dtype=np.float32)
    for r in range(W):
        wl.fill(2, r, 0, n, host[r * stride:r * stride + n])
    s = torch.cuda.Stream()
    dev = torch.device("cuda:0")
    with torch.cuda.stream(s):
        grads = torch.from_numpy(host).to(dev)
        nc, d_off = H.plan_device([n], 4, dev, stream=s)
        ws = _ws(W, stride, nc, dev)
        out = torch.empty(n, dtype=torch.float32, device=dev)
        gq.gq_fused_allreduce_sim_pipelined(grads, W, stride, d_off, nc, 1024.0, "ring", out, ws, stream=s)
        assert gq.gq_get_error(s) == gq.GQ_OK
    want = oracle.fused(host, W, stride, oracle.plan_chunks([n], 4), oracle.RING, 1024.0)[0]
    H.assert_bits_equal(out.cpu().numpy(), want, "output")


def test_pipe_workload4_bert_fp16_sampled():
    """W = 16 BERT-Large fp16 shapes (335,141,888 elements per rank), loss scale 65536, ring:
    bucket-boundary, first, last and random chunks against the oracle."""
    W = 16
    dev = torch.device("cuda:0")
    sizes, _ = wl.tensor_layout(4)
    n = int(sizes.sum())
    _, buckets = gq.gq_plan_buckets(sizes, 2)
    stride = gq.row_stride(n, 2)
    grads = torch.empty(W * stride, dtype=torch.float16, device=dev)
    tmp = np.zeros(stride, dtype=np.float16)
    for r in range(W):
        wl.fill(4, r, 0, n, tmp[:n])
        grads[r * stride:(r + 1) * stride].copy_(torch.from_numpy(tmp))
    nc, d_off = H.plan_device(list(buckets), 2, dev)
    off = d_off.cpu().numpy()
    out = torch.empty(n, dtype=torch.float32, device=dev)
    scales = torch.empty(W * nc, dtype=torch.float32, device=dev)
    ws = _ws(W, stride, nc, dev)
    gq.gq_fused_allreduce_sim_pipelined(grads, W, stride, d_off, nc, 65536.0, "ring", out, ws, None, scales)
    assert gq.gq_get_error() == gq.GQ_OK
    out_h = out.cpu().numpy()
    scales_h = scales.cpu().numpy().reshape(W, nc)
    del grads, ws

    def rows(lo, hi):
        return np.stack([wl.fill(4, r, lo, hi) for r in range(W)])

    starts = np.concatenate([[0], np.cumsum(buckets)[:-1]])
    bucket_first = [int(np.searchsorted(off, s)) for s in starts]
    chunks = sorted(set(H.sample_chunks(nc, 40, 5)) | set(bucket_first))
    H.compare_sampled(rows, W, off, chunks, oracle.RING, 65536.0, out_h, None, scales_h, stride)


def test_pipe_copy_wait_runs_out_and_is_reported():
    """Failure detection without a GPU fault: the first bulk copy of every CTA is told to expect 16
    bytes more than it delivers, so its wait gives up after the (2 ms) limit; the call reports
    GQ_ERR_TIMEOUT, the context stays usable, and a call on a re-zeroed workspace is bit-exact."""
    W, n = 8, 1 << 20
    host, stride = wl.rows(2, W, n)
    dev = torch.device("cuda:0")
    grads = torch.from_numpy(host).to(dev)
    nc, d_off = H.plan_device([n], 4, dev)
    ws = _ws(W, stride, nc, dev)
    out = torch.empty(n, dtype=torch.float32, device=dev)
    assert gq.gq_get_error() == gq.GQ_OK
    try:
        gq.gq_testing_inject_copy_stall(16, 2_000_000)
        gq.gq_fused_allreduce_sim_pipelined(grads, W, stride, d_off, nc, 1.0, "ring", out, ws)
        assert gq.gq_get_error() == gq.GQ_ERR_TIMEOUT
    finally:
        gq.gq_testing_inject_copy_stall(0, 0)
    ws.zero_()
    gq.gq_fused_allreduce_sim_pipelined(grads, W, stride, d_off, nc, 1.0, "ring", out, ws)
    assert gq.gq_get_error() == gq.GQ_OK
    want = oracle.fused(host, W, stride, d_off.cpu().numpy(), oracle.RING)[0]
    H.assert_bits_equal(out.cpu().numpy(), want, "output after the timeout")


@pytest.mark.parametrize("world", [3])
def test_pipe_sharded_table(world):
    """The multi-GPU split run on one GPU: each shard's sub-table (global offsets) through the
    pipelined call and the two-kernel path writes its own output range; together they are the
    unsplit result, bit for bit."""
    from dp_gradient_bucket_gb300 import shard
    W = 8
    buckets = [5, 65535, 131075, 7, 32769 * 3 + 1, 3, 49152]
    off = oracle.plan_chunks(buckets, 4)
    n = int(off[-1])
    stride = gq.row_stride(n, 4)
    host = np.zeros(W * stride, dtype=np.float32)
    for r in range(W):
        wl.fill(2, r, 0, n, host[r * stride:r * stride + n])
    dev = torch.device("cuda:0")
    grads = torch.from_numpy(host).to(dev)
    want = oracle.fused(host, W, stride, off, oracle.RING)[0]
    out = torch.zeros(n, dtype=torch.float32, device=dev)
    out2 = torch.zeros(n, dtype=torch.float32, device=dev)
    codes = torch.zeros(W * stride, dtype=torch.int8, device=dev)
    for rank in range(world):
        sub, k = shard.shard_table(off, world, rank)
        if k == 0:
            continue
        d_sub = torch.from_numpy(sub).to(dev)
        ws = _ws(W, stride, k, dev)
        gq.gq_fused_allreduce_sim_pipelined(grads, W, stride, d_sub, k, 1.0, "ring", out, ws)
        scales = torch.zeros(W * k, dtype=torch.float32, device=dev)
        gq.gq_quantize(grads, W, stride, d_sub, k, 1.0, codes, scales)
        gq.gq_reduce_dequant(codes, scales, W, stride, d_sub, k, "ring", out2)
    assert gq.gq_get_error() == gq.GQ_OK
    H.assert_bits_equal(out.cpu().numpy(), want, "pipelined, sharded")
    H.assert_bits_equal(out2.cpu().numpy(), want, "two-kernel, sharded")
