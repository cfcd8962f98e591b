"""Helpers for the GPU parity tests: run the library through the binding with guard
canaries around every output buffer, and compare with the oracle."""
import numpy as np
import torch

import dp_gradient_bucket_gb300 as gq
import oracle

GUARD = 64          # elements of guard before and after each output
CANARY_F32 = 0x7fa5a5a5   # a NaN pattern no kernel writes
CANARY_I8 = -91           # 0xa5


def f32_canary(n, dev):
    return torch.full((n + 2 * GUARD,), CANARY_F32, dtype=torch.int32, device=dev).view(torch.float32)


def i8_canary(n, dev):
    return torch.full((n + 2 * GUARD,), CANARY_I8, dtype=torch.int8, device=dev)


def inner(buf, n):
    return buf[GUARD:GUARD + n]


def guards_intact(buf, n):
    b = buf.view(torch.int32) if buf.dtype == torch.float32 else buf
    want = CANARY_F32 if buf.dtype == torch.float32 else CANARY_I8
    head, tail = b[:GUARD], b[GUARD + n:]
    return bool((head == want).all()) and bool((tail == want).all())


def plan_device(bucket_elems, eb, dev, stream=None, scope=None, chunk_bytes=None):
    if scope is None and chunk_bytes is None:
        nc = gq.gq_plan_chunks(bucket_elems, eb)
        offsets = torch.full((nc + 1,), -1, dtype=torch.int64, device=dev)
        gq.gq_plan_chunks(bucket_elems, eb, offsets, stream=stream)
        return nc, offsets
    scope = scope or "chunk"
    chunk_bytes = chunk_bytes or gq.GQ_CHUNK_SIZE
    nc = gq.gq_plan_chunks_ex(bucket_elems, eb, scope, chunk_bytes)
    offsets = torch.full((nc + 1,), -1, dtype=torch.int64, device=dev)
    gq.gq_plan_chunks_ex(bucket_elems, eb, scope, chunk_bytes, offsets, stream=stream)
    return nc, offsets


def run(host_rows, W, stride, bucket_elems, order, loss_scale=1.0, mode="fused", dev="cuda:0",
        offsets=None, want_codes=True, scope=None, chunk_bytes=None):
    """Runs the path on the GPU.  Returns (out, codes, scales, offsets_host, status) as numpy."""
    dev = torch.device(dev)
    eb = host_rows.dtype.itemsize
    grads = torch.from_numpy(host_rows).to(dev)
    if offsets is None:
        nc, d_off = plan_device(bucket_elems, eb, dev, scope=scope, chunk_bytes=chunk_bytes)
    else:
        d_off = torch.from_numpy(np.ascontiguousarray(offsets, dtype=np.int64)).to(dev)
        nc = len(offsets) - 1
    n_total = int(d_off[-1].item()) if offsets is None else max(int(offsets[-1]), 0)
    # at least one group, so an empty problem still passes a real (non-null) output pointer
    n_out = max(n_total, stride, 4) if offsets is not None else max(n_total, 4)
    out_buf = f32_canary(n_out, dev)
    codes_buf = i8_canary(W * stride, dev)
    scales_buf = f32_canary(W * nc, dev)
    out, codes, scales = inner(out_buf, n_out), inner(codes_buf, W * stride), inner(scales_buf, W * nc)
    ws = None
    if mode == "fused":
        gq.gq_fused_allreduce_sim(grads, W, stride, d_off, nc, loss_scale, order, out,
                                  codes if want_codes else None, scales if want_codes else None)
    elif mode == "fused_ws":
        ws = torch.zeros(gq.gq_fused_workspace_bytes(nc, W) // 4, dtype=torch.int32, device=dev)
        for _ in range(2):  # a second call on the same workspace: it must have been left zeroed
            gq.gq_fused_allreduce_sim_ws(grads, W, stride, d_off, nc, loss_scale, order, out, ws,
                                         codes if want_codes else None, scales if want_codes else None)
    elif mode == "pipe":
        ws = torch.zeros(gq.gq_pipelined_workspace_bytes(W, stride, nc), dtype=torch.uint8, device=dev)
        for _ in range(2):  # a second call on the same workspace: counters reset, epoch advanced
            gq.gq_fused_allreduce_sim_pipelined(grads, W, stride, d_off, nc, loss_scale, order, out, ws,
                                                codes if want_codes else None, scales if want_codes else None)
    else:
        gq.gq_quantize(grads, W, stride, d_off, nc, loss_scale, codes, scales)
        gq.gq_reduce_dequant(codes, scales, W, stride, d_off, nc, order, out)
    status = gq.gq_get_error()
    if ws is not None and mode == "fused_ws":
        # the queue head and exit count are back at zero for the next call
        assert int(ws[0].item()) == 0 and int(ws[1].item()) == 0, "workspace header not reset"
    if ws is not None and mode == "pipe":
        assert pipe_header(ws) == (0, 0, 0, 2), "workspace header after two calls: %r" % (pipe_header(ws),)
    assert guards_intact(out_buf, n_out), "write outside the output buffer"
    assert guards_intact(codes_buf, W * stride), "write outside the codes buffer"
    assert guards_intact(scales_buf, W * nc), "write outside the scales buffer"
    return (out.cpu().numpy(), codes.cpu().numpy(), scales.cpu().numpy().reshape(W, nc),
            d_off.cpu().numpy(), status)


def pipe_header(ws):
    """(quantise counter, reduce counter, exit count, launch epoch) of a pipelined workspace."""
    h = ws[:24].cpu().numpy()
    return (int(h[0:8].view(np.uint64)[0]), int(h[8:16].view(np.uint64)[0]), int(h[16:20].view(np.uint32)[0]),
            int(h[20:24].view(np.uint32)[0]))


def assert_bits_equal(got, want, what):
    g = np.ascontiguousarray(got).view(np.uint32)
    w = np.ascontiguousarray(want).view(np.uint32)
    if not np.array_equal(g, w):
        bad = np.nonzero(g != w)[0]
        i = bad[0]
        raise AssertionError("%s: %d of %d differ; first at %d: got %r (0x%08x) want %r (0x%08x)" % (
            what, len(bad), len(w), i, got.reshape(-1)[i], g.reshape(-1)[i], want.reshape(-1)[i], w.reshape(-1)[i]))


def compare_full(host_rows, W, stride, offsets, order, loss_scale, out, codes, scales, check_codes=True):
    """The whole problem against the oracle, bit for bit (codes, scales, output)."""
    want, wcodes, wscales, nf = oracle.fused(host_rows, W, stride, offsets, order, loss_scale)
    n = int(offsets[-1])
    assert_bits_equal(out[:n], want, "output")
    assert_bits_equal(scales, wscales, "scales")
    if check_codes:
        for r in range(W):
            c = codes[r * stride:r * stride + n]
            assert np.array_equal(c, wcodes[r * stride:r * stride + n]), "codes of rank %d" % r
    return nf


def sample_chunks(num_chunks, k, seed):
    rng = np.random.default_rng(seed)
    pick = {0, num_chunks - 1, num_chunks // 2}
    pick |= set(int(x) for x in rng.integers(0, num_chunks, k))
    return sorted(pick)


def compare_sampled(get_rows, W, offsets, chunks, order, loss_scale, out, codes, scales, stride):
    """Chosen chunks against the oracle run on just those chunks (chunks are independent:
    a chunk's scale and ring segments depend on that chunk alone)."""
    for j in chunks:
        lo, hi = int(offsets[j]), int(offsets[j + 1])
        n = hi - lo
        sub = get_rows(lo, hi)   # [W, n] host array of the chunk's elements
        sstride = gq.row_stride(max(n, 1), sub.dtype.itemsize)
        rows = np.zeros(W * sstride, dtype=sub.dtype)
        for r in range(W):
            rows[r * sstride:r * sstride + n] = sub[r]
        want, wcodes, wscales, _ = oracle.fused(rows, W, sstride, np.array([0, n]), order, loss_scale)
        assert_bits_equal(out[lo:hi], want, "output of chunk %d" % j)
        assert_bits_equal(scales[:, j], wscales[:, 0], "scales of chunk %d" % j)
        if codes is not None:
            for r in range(W):
                assert np.array_equal(codes[r * stride + lo:r * stride + hi], wcodes[r * sstride:r * sstride + n]), \
                    "codes of chunk %d rank %d" % (j, r)
