"""ctypes front end of the CPU oracle.

TEST INFRASTRUCTURE ONLY: the tests, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference legs may import this package; the library in
dp_gradient_bucket_gb300/ never does.  Arrays are numpy; nothing here computes any
step of the method (the arithmetic is all in oracle.cpp).
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32, F16 = 0, 1
SEQ, RING, TREE = 0, 1, 2
HIER_BASE = 0x100


def HIER(L):
    """Order code of the hierarchical order with nodes of L ranks (same encoding as gq.h)."""
    return HIER_BASE + int(L)

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        L.oracle_bucket_chunks.argtypes = [i64, i64, p]
        L.oracle_bucket_chunks.restype = i64
        L.oracle_plan_chunks.argtypes = [p, i64, i64, p, i64]
        L.oracle_plan_chunks.restype = i64
        L.oracle_bucket_chunks_sized.argtypes = [i64, i64, i64, p]
        L.oracle_bucket_chunks_sized.restype = i64
        L.oracle_plan_chunks_ex.argtypes = [p, i64, i64, ctypes.c_int, i64, p, i64]
        L.oracle_plan_chunks_ex.restype = i64
        L.oracle_assign_buckets.argtypes = [p, i64, i64, i64, p, p, i64]
        L.oracle_assign_buckets.restype = i64
        L.oracle_quantize.argtypes = [p, ctypes.c_int, ctypes.c_int, i64, p, i64, ctypes.c_float, p, p]
        L.oracle_quantize.restype = i64
        L.oracle_reduce.argtypes = [p, p, ctypes.c_int, i64, p, i64, ctypes.c_int, p]
        L.oracle_reduce.restype = None
        L.oracle_reduce_hier.argtypes = [p, p, ctypes.c_int, i64, p, i64, ctypes.c_int, p]
        L.oracle_reduce_hier.restype = ctypes.c_int
        L.oracle_amp_update_scale.argtypes = [p, p, ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_int32]
        L.oracle_amp_update_scale.restype = None
        L.oracle_half_to_float.argtypes = [ctypes.c_uint16]
        L.oracle_half_to_float.restype = ctypes.c_float
        _lib = L
    return _lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def bucket_chunks(n, eb):
    """(count, piece length) of dynamic_chunk on one bucket of n elements."""
    c = ctypes.c_int64(0)
    k = lib().oracle_bucket_chunks(int(n), int(eb), ctypes.byref(c))
    return int(k), int(c.value)


def bucket_chunks_sized(n, eb, chunk_size):
    """(count, piece length) of dynamic_chunk with base chunk size chunk_size bytes."""
    c = ctypes.c_int64(0)
    k = lib().oracle_bucket_chunks_sized(int(n), int(eb), int(chunk_size), ctypes.byref(c))
    return int(k), int(c.value)


SCOPE_CHUNK, SCOPE_BUCKET, SCOPE_TENSOR = 0, 1, 2


def plan_chunks_ex(elems, eb, scope=SCOPE_CHUNK, chunk_size=128 * 1024):
    """int64 offsets[num_chunks + 1] for entries (buckets or tensors) laid end to end."""
    be = np.ascontiguousarray(elems, dtype=np.int64)
    total = lib().oracle_plan_chunks_ex(_ptr(be), len(be), int(eb), int(scope), int(chunk_size), None, 0)
    if total < 0:
        raise ValueError("bad plan arguments")
    off = np.empty(total + 1, dtype=np.int64)
    lib().oracle_plan_chunks_ex(_ptr(be), len(be), int(eb), int(scope), int(chunk_size), _ptr(off), len(off))
    return off


def plan_chunks(bucket_elems, eb):
    """int64 offsets[num_chunks + 1] for buckets laid end to end."""
    be = np.ascontiguousarray(bucket_elems, dtype=np.int64)
    total = lib().oracle_plan_chunks(_ptr(be), len(be), int(eb), None, 0)
    if total < 0:
        raise ValueError("negative bucket size")
    off = np.empty(total + 1, dtype=np.int64)
    lib().oracle_plan_chunks(_ptr(be), len(be), int(eb), _ptr(off), len(off))
    return off


def assign_buckets(tensor_elems, eb, cap_bytes=25 * 1024 * 1024):
    """(bucket_of_tensor[int64], bucket_elems[int64]) by the greedy list-order rule."""
    te = np.ascontiguousarray(tensor_elems, dtype=np.int64)
    bot = np.empty(max(len(te), 1), dtype=np.int64)
    be = np.empty(max(len(te), 1), dtype=np.int64)
    nb = lib().oracle_assign_buckets(_ptr(te), len(te), int(eb), int(cap_bytes), _ptr(bot), _ptr(be), len(be))
    if nb < 0:
        raise RuntimeError("bucket capacity exceeded")
    return bot[:len(te)].copy(), be[:nb].copy()


def quantize(grads, W, rank_stride, offsets, loss_scale=1.0):
    """grads: float32 or float16 array holding W rows of rank_stride elements.
    Returns (codes int8 [W*rank_stride], scales f32 [W, num_chunks], nonfinite count)."""
    g = np.ascontiguousarray(grads)
    if g.dtype == np.float32:
        dt = F32
    elif g.dtype == np.float16:
        dt = F16
    else:
        raise TypeError(g.dtype)
    g = g.reshape(-1)
    assert g.size >= W * rank_stride
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    nc = len(off) - 1
    codes = np.zeros(W * rank_stride, dtype=np.int8)
    scales = np.zeros((W, nc), dtype=np.float32)
    nf = lib().oracle_quantize(_ptr(g), dt, int(W), int(rank_stride), _ptr(off), nc,
                               float(loss_scale), _ptr(codes), _ptr(scales))
    return codes, scales, int(nf)


def reduce(codes, scales, W, rank_stride, offsets, order):
    """Mean of the dequantised codes over W ranks in the given order -> f32 [offsets[-1]]."""
    c = np.ascontiguousarray(codes, dtype=np.int8).reshape(-1)
    s = np.ascontiguousarray(scales, dtype=np.float32)
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    nc = len(off) - 1
    assert s.size == W * nc and c.size >= W * rank_stride
    out = np.zeros(int(off[-1]), dtype=np.float32)
    if order > HIER_BASE:
        rc = lib().oracle_reduce_hier(_ptr(c), _ptr(s), int(W), int(rank_stride), _ptr(off), nc,
                                      int(order) - HIER_BASE, _ptr(out))
        if rc != 0:
            raise ValueError("node size %d does not divide W = %d" % (order - HIER_BASE, W))
        return out
    lib().oracle_reduce(_ptr(c), _ptr(s), int(W), int(rank_stride), _ptr(off), nc, int(order), _ptr(out))
    return out


def fused(grads, W, rank_stride, offsets, order, loss_scale=1.0):
    """quantize then reduce: (out, codes, scales, nonfinite)."""
    codes, scales, nf = quantize(grads, W, rank_stride, offsets, loss_scale)
    return reduce(codes, scales, W, rank_stride, offsets, order), codes, scales, nf


def half_to_float(bits):
    return float(lib().oracle_half_to_float(int(bits)))


def amp_update_scale(scale, tracker, found_inf, growth=2.0, backoff=0.5, interval=2000):
    """One GradScaler update step; returns (scale float32, tracker int)."""
    sc = np.array([scale], dtype=np.float32)
    tr = np.array([tracker], dtype=np.int32)
    lib().oracle_amp_update_scale(_ptr(sc), _ptr(tr), float(np.float32(found_inf)), float(growth), float(backoff),
                                  int(interval))
    return sc[0], int(tr[0])
