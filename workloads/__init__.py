"""Seeded synthetic workloads (inputs only; none of the method's arithmetic).

Five workloads, each W virtual ranks of flat gradient rows:
  1  W=2, 262,144 fp32 per rank, N(0, 1e-3), sequential order
  2  W=8, one 25 MiB fp32 DDP bucket (6,553,600) per rank, Laplace(0, 1e-4) with 30%
     exact zeros and 0.1% outliers x100, ring order
  3  W=8, ResNet-152-sized list (60,192,808 fp32 per rank, log-uniform tensor sizes
     64..2,359,296, per-tensor sigma log-uniform 1e-6..1e-2), ring order
  4  W=16, BERT-Large fp16 shapes (335,141,888 per rank) x 65536 loss scale, ring order
  5  W=8 fp32 size sweep 4 KiB..1 GiB plus ragged sizes, with adversarial chunks
Seeds are 0x67510000 + workload id; rank r is sub-stream r.
"""
import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "libwlgen.so")
SRC = os.path.join(HERE, "gen.cpp")

CONFIGS = {
    1: dict(W=2, dtype="f32", order="seq", loss_scale=1.0, n=262144),
    2: dict(W=8, dtype="f32", order="ring", loss_scale=1.0, n=6553600),
    3: dict(W=8, dtype="f32", order="ring", loss_scale=1.0, n=60192808),
    4: dict(W=16, dtype="f16", order="ring", loss_scale=65536.0, n=335141888),
    5: dict(W=8, dtype="f32", order="ring", loss_scale=1.0, n=None),
}

SWEEP_SIZES = ([2 ** k for k in range(10, 29)]
               + [2 ** k + d for k in (12, 16, 20, 24) for d in (-1, 3, 17)] + [1000003])

_lib = None


def seed(cfg):
    return 0x67510000 + int(cfg)


def build(force=False):
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    subprocess.check_call(["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                           "-pthread", SRC, "-o", tmp])
    os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        i64, p = ctypes.c_int64, ctypes.c_void_p
        L.wl_tensor_layout.argtypes = [ctypes.c_int, ctypes.c_uint64, p, p, i64]
        L.wl_tensor_layout.restype = i64
        L.wl_fill.argtypes = [ctypes.c_int, ctypes.c_uint64, ctypes.c_int, i64, i64, p, ctypes.c_int]
        L.wl_fill.restype = ctypes.c_int
        L.wl_adversarial.argtypes = [ctypes.c_uint64, ctypes.c_int, i64, p, i64, p]
        L.wl_adversarial.restype = ctypes.c_int
        _lib = L
    return _lib


def threads():
    return max(1, min(32, os.cpu_count() or 1))


def tensor_layout(cfg):
    """(sizes int64[T], sigmas f64[T]) of workload 3 or 4; None for the others."""
    nt = lib().wl_tensor_layout(cfg, seed(cfg), None, None, 0)
    if nt < 0:
        return None
    sizes = np.empty(nt, dtype=np.int64)
    sig = np.empty(nt, dtype=np.float64)
    lib().wl_tensor_layout(cfg, seed(cfg), sizes.ctypes.data, sig.ctypes.data, nt)
    return sizes, sig


def np_dtype(cfg):
    return np.float16 if CONFIGS[cfg]["dtype"] == "f16" else np.float32


def fill(cfg, rank, i0, i1, out=None):
    """Elements [i0, i1) of rank `rank` of workload cfg (float32, or float16 for cfg 4)."""
    dt = np_dtype(cfg)
    if out is None:
        out = np.empty(i1 - i0, dtype=dt)
    assert out.dtype == dt and out.size >= i1 - i0 and out.flags.c_contiguous
    rc = lib().wl_fill(cfg, seed(cfg), int(rank), int(i0), int(i1), out.ctypes.data, threads())
    if rc != 0:
        raise ValueError("unknown workload %r" % cfg)
    return out


def row_stride(n, elem_bytes):
    """Row stride (elements) that starts every rank's row on a 16-byte boundary."""
    per = 16 // elem_bytes
    return max(per, -(-n // per) * per)


def rows(cfg, W, n, stride=None, out=None):
    """W rows of `stride` elements (padding zero), elements [0, n) of each rank."""
    dt = np_dtype(cfg)
    if stride is None:
        stride = row_stride(n, np.dtype(dt).itemsize)
    if out is None:
        out = np.zeros(W * stride, dtype=dt)
    for r in range(W):
        fill(cfg, r, 0, n, out[r * stride:r * stride + n])
    return out, stride


def adversarial(rows_f32, W, stride, offsets):
    """Overwrite chunks 0..4 of every row with workload 5's adversarial patterns."""
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    assert rows_f32.dtype == np.float32 and rows_f32.flags.c_contiguous
    rc = lib().wl_adversarial(seed(5), int(W), int(stride), off.ctypes.data, len(off) - 1,
                              rows_f32.ctypes.data)
    if rc != 0:
        raise ValueError("adversarial patterns need at least five chunks")
    return rows_f32
