"""Seeded synthetic inputs for the Q8_0 x Q8_0 matmul workloads.

A module of its own: both the oracle's tests and the CUDA path's tests and
benchmark draw their inputs here, and it holds none of the method's
arithmetic (no quantisation, no dot products).  The numbers come from the C
file ``q8gen.c`` beside this one (counter-based SplitMix64), so every value is
a pure function of (seed, stream, index) and is the same on x86_64 and
aarch64.  The distributions follow the workloads named for the dense
projections and routed experts of the ds4 engine (attn_q_a / q_b /
output_a / output_b, shared and routed experts).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q8gen.c")
_LIB = os.path.join(_HERE, "libq8gen.so")
_lock = threading.Lock()
_lib = None

BLOCK = 32
BLOCK_BYTES = 34

# Stream ids: one per tensor role, so inputs never overlap.
STREAM_W = 1
STREAM_X = 2
STREAM_ROUTE = 3


def build(force: bool = False) -> str:
    """Compile libq8gen.so in place (gcc, OpenMP) when missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC",
                               "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i32, u32, dbl, vp = (ctypes.c_uint64, ctypes.c_int32, ctypes.c_uint32,
                                      ctypes.c_double, ctypes.c_void_p)
            lib.q8g_weights.argtypes = [vp, u64, u64, u64, u64, dbl, dbl]
            lib.q8g_kq_weights.argtypes = [vp, u64, u64, i32, u64, u64, dbl, dbl, dbl, dbl]
            lib.q8g_kq_weights.restype = ctypes.c_int
            lib.q8g_normal.argtypes = [vp, u64, u64, u64, dbl, dbl]
            lib.q8g_route_uniform.argtypes = [vp, u64, u32, u32, u64, u64]
            lib.q8g_route_zipf.argtypes = [vp, u64, u32, u32, dbl, u64, u64]
            for f in (lib.q8g_weights, lib.q8g_normal, lib.q8g_route_uniform, lib.q8g_route_zipf):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def weights(rows: int, in_dim: int, seed: int = 0, stream: int = STREAM_W,
            d_lo: float = 1e-3, d_hi: float = 1e-2, out: np.ndarray | None = None) -> np.ndarray:
    """Raw Q8_0 rows: uint8 array of shape [rows, in_dim/32*34]."""
    assert in_dim % BLOCK == 0
    nbytes = rows * (in_dim // BLOCK) * BLOCK_BYTES
    if out is None:
        out = np.empty((rows, (in_dim // BLOCK) * BLOCK_BYTES), dtype=np.uint8)
    assert out.dtype == np.uint8 and out.flags.c_contiguous and out.nbytes == nbytes
    rc = _load().q8g_weights(_ptr(out), rows, in_dim, seed, stream, d_lo, d_hi)
    assert rc == 0
    return out


KQ_BLOCK = 256
KQ_BYTES = {2: 84, 4: 144}      # Q2_K, Q4_K
# d and dmin ranges (binary16 normal numbers) that give weights of a few hundredths
KQ_SCALES = {2: (5e-4, 2e-3, 5e-4, 2e-3), 4: (6.2e-5, 1.5e-4, 6.2e-5, 1.5e-4)}


def kq_weights(rows: int, in_dim: int, fmt: int, seed: int = 0, stream: int = STREAM_W,
               scales=None, out: np.ndarray | None = None) -> np.ndarray:
    """Raw K-quant rows (fmt 2: Q2_K, 4: Q4_K): uint8 [rows, in_dim/256*block bytes]."""
    assert in_dim % KQ_BLOCK == 0 and fmt in KQ_BYTES
    shape = (rows, in_dim // KQ_BLOCK * KQ_BYTES[fmt])
    if out is None:
        out = np.empty(shape, dtype=np.uint8)
    assert out.dtype == np.uint8 and out.flags.c_contiguous and out.size == shape[0] * shape[1]
    d_lo, d_hi, m_lo, m_hi = scales or KQ_SCALES[fmt]
    assert _load().q8g_kq_weights(_ptr(out), rows, in_dim, fmt, seed, stream, d_lo, d_hi, m_lo, m_hi) == 0
    return out


def normal(shape, seed: int = 0, stream: int = STREAM_X, p_out: float = 0.0,
           out_scale: float = 20.0, out: np.ndarray | None = None) -> np.ndarray:
    """float32 N(0,1) array; each element scaled by out_scale with probability p_out."""
    if out is None:
        out = np.empty(shape, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous
    rc = _load().q8g_normal(_ptr(out), out.size, seed, stream, p_out, out_scale)
    assert rc == 0
    return out


def route_uniform(n_tok: int, k: int, n_expert: int, seed: int = 0,
                  stream: int = STREAM_ROUTE) -> np.ndarray:
    """int32 [n_tok, k]: k distinct experts per token, uniform."""
    ids = np.empty((n_tok, k), dtype=np.int32)
    assert _load().q8g_route_uniform(_ptr(ids), n_tok, k, n_expert, seed, stream) == 0
    return ids


def route_zipf(n_tok: int, k: int, n_expert: int, s: float = 1.1, seed: int = 0,
               stream: int = STREAM_ROUTE) -> np.ndarray:
    """int32 [n_tok, k]: k distinct experts per token, Zipf(s) over ranks (rank r -> expert r-1)."""
    ids = np.empty((n_tok, k), dtype=np.int32)
    assert _load().q8g_route_zipf(_ptr(ids), n_tok, k, n_expert, s, seed, stream) == 0
    return ids
