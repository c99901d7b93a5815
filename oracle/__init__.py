"""CPU oracle for the Q8_0 x Q8_0 matmul -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never does, and there is no CPU fallback through it.

The arithmetic lives in the plain C file ``q8_oracle.c`` beside this one
(built with gcc, no fast-math, no FMA contraction); this wrapper only
marshals numpy arrays.  Every function is pinned by tests that do not use the
oracle's own code (see ``tests/test_oracle_pins.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "q8_oracle.c")
_LIB = os.path.join(_HERE, "libq8oracle.so")
CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
_lock = threading.Lock()
_lib = None

QK = 32
QBYTES = 34
QKK = 256           # weights per K-quant block and values per Q8_K block
KQ_Q2, KQ_Q4 = 2, 4  # K-quant formats: Q2_K (84-byte blocks), Q4_K (144-byte blocks)


def compile_lib(src: str, dst: str) -> str:
    """Compile an oracle source file into a shared library (used by build() and the mutation tests)."""
    tmp = dst + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, src, "-lm"])
    os.replace(tmp, dst)
    return dst


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_lib(SOURCE, _LIB)
    return _LIB


class Oracle:
    """ctypes view of one compiled oracle library (the real one, or a test mutant)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        vp, u64, u32, i32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int
        lib.q8o_f32_to_f16.argtypes = [ctypes.c_float]
        lib.q8o_f32_to_f16.restype = ctypes.c_uint16
        lib.q8o_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.q8o_f16_to_f32.restype = ctypes.c_float
        lib.q8o_quantize.argtypes = [vp, vp, u64, u64]
        lib.q8o_matmul.argtypes = [vp, vp, vp, u64, u64, vp, u64]
        lib.q8o_matmul_sample.argtypes = [vp, vp, vp, u64, u64, vp, u64, vp, vp, u64]
        lib.q8o_moe.argtypes = [vp, vp, vp, u32, u64, vp, u32, u64, u64, vp, i32, u64]
        lib.q8o_moe_sample.argtypes = [vp, vp, vp, u32, u64, vp, u32, u64, u64, vp, i32, u64,
                                       vp, vp, u64]
        lib.q8o_swiglu.argtypes = [vp, vp, vp, u64, ctypes.c_float]
        lib.q8o_swiglu.restype = None
        lib.q8o_combine.argtypes = [vp, vp, vp, vp, u64, u32, u64]
        lib.q8o_combine.restype = None
        lib.q8o_moe_ffn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, u32, u64, u64, vp, vp, u32,
                                    u64, u64, u64, ctypes.c_float, vp, u64]
        lib.q8o_rmsnorm_quantize.argtypes = [vp, vp, vp, vp, u64, u64, ctypes.c_double]
        lib.q8o_kq_block_bytes.argtypes = [i32]
        lib.q8o_kq_block_bytes.restype = u64
        lib.q8o_kq_dequant.argtypes = [vp, vp, i32, u64, u64]
        lib.q8o_quantize_q8k.argtypes = [vp, vp, vp, u64, u64]
        lib.q8o_kq_matmul_q.argtypes = [vp, vp, vp, i32, u64, u64, vp, vp, u64]
        lib.q8o_kq_moe.argtypes = [vp, vp, vp, i32, u32, u64, vp, u32, u64, u64, vp, vp, i32, u64]
        for f in (lib.q8o_quantize, lib.q8o_matmul, lib.q8o_matmul_sample, lib.q8o_moe,
                  lib.q8o_moe_sample, lib.q8o_moe_ffn, lib.q8o_rmsnorm_quantize, lib.q8o_kq_dequant,
                  lib.q8o_quantize_q8k, lib.q8o_kq_matmul_q, lib.q8o_kq_moe):
            f.restype = ctypes.c_int
        self.lib = lib

    # -- binary16 ------------------------------------------------------------
    def f32_to_f16(self, v: float) -> int:
        return int(self.lib.q8o_f32_to_f16(float(v)))

    def f16_to_f32(self, h: int) -> float:
        return float(self.lib.q8o_f16_to_f32(int(h)))

    # -- quantiser -------------------------------------------------------------
    def quantize(self, x: np.ndarray) -> np.ndarray:
        """x float32 [n_tok, in_dim] -> uint8 [n_tok, in_dim/32*34] canonical blocks."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim == 1:
            x = x[None, :]
        n_tok, in_dim = x.shape
        xq = np.empty((n_tok, in_dim // QK * QBYTES), dtype=np.uint8)
        rc = self.lib.q8o_quantize(xq.ctypes.data, x.ctypes.data, in_dim, n_tok)
        if rc != 0:
            raise ValueError("oracle quantize: bad dims")
        return xq

    # -- matmul ------------------------------------------------------------------
    def matmul_q(self, W: np.ndarray, xq: np.ndarray, in_dim: int, out_dim: int, n_tok: int):
        """Returns (out float32 [n_tok, out_dim], bound float64 [n_tok, out_dim])."""
        W = np.ascontiguousarray(W, dtype=np.uint8)
        xq = np.ascontiguousarray(xq, dtype=np.uint8)
        assert W.nbytes == out_dim * in_dim // QK * QBYTES
        assert xq.nbytes == n_tok * in_dim // QK * QBYTES
        out = np.empty((n_tok, out_dim), dtype=np.float32)
        bound = np.empty((n_tok, out_dim), dtype=np.float64)
        rc = self.lib.q8o_matmul(out.ctypes.data, bound.ctypes.data, W.ctypes.data, in_dim,
                                 out_dim, xq.ctypes.data, n_tok)
        if rc != 0:
            raise ValueError("oracle matmul: bad dims")
        return out, bound

    def matmul(self, W: np.ndarray, x: np.ndarray, out_dim: int):
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim == 1:
            x = x[None, :]
        n_tok, in_dim = x.shape
        return self.matmul_q(W, self.quantize(x), in_dim, out_dim, n_tok)

    def matmul_sample(self, W, xq, in_dim, out_dim, n_tok, tok, row):
        tok = np.ascontiguousarray(tok, dtype=np.int64)
        row = np.ascontiguousarray(row, dtype=np.int64)
        out = np.empty(tok.size, dtype=np.float32)
        bound = np.empty(tok.size, dtype=np.float64)
        rc = self.lib.q8o_matmul_sample(out.ctypes.data, bound.ctypes.data,
                                        np.ascontiguousarray(W).ctypes.data, in_dim, out_dim,
                                        np.ascontiguousarray(xq).ctypes.data, n_tok,
                                        tok.ctypes.data, row.ctypes.data, tok.size)
        if rc != 0:
            raise ValueError("oracle matmul_sample: bad arguments")
        return out, bound

    # -- routed experts ------------------------------------------------------------
    def moe(self, W_experts, n_expert, expert_stride, ids, in_dim, out_dim, xq, x_per_pair, n_tok):
        """Returns (out [n_tok*k, out_dim], bound, flag)."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        k = ids.size // n_tok if n_tok else 1
        out = np.empty((n_tok * k, out_dim), dtype=np.float32)
        bound = np.empty((n_tok * k, out_dim), dtype=np.float64)
        rc = self.lib.q8o_moe(out.ctypes.data, bound.ctypes.data,
                              np.ascontiguousarray(W_experts).ctypes.data, n_expert, expert_stride,
                              ids.ctypes.data, k, in_dim, out_dim,
                              np.ascontiguousarray(xq).ctypes.data, int(x_per_pair), n_tok)
        if rc < 0:
            raise ValueError("oracle moe: bad dims")
        return out, bound, rc

    def moe_sample(self, W_experts, n_expert, expert_stride, ids, in_dim, out_dim, xq,
                   x_per_pair, n_tok, pair, row):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        k = ids.size // n_tok
        pair = np.ascontiguousarray(pair, dtype=np.int64)
        row = np.ascontiguousarray(row, dtype=np.int64)
        out = np.empty(pair.size, dtype=np.float32)
        bound = np.empty(pair.size, dtype=np.float64)
        rc = self.lib.q8o_moe_sample(out.ctypes.data, bound.ctypes.data,
                                     np.ascontiguousarray(W_experts).ctypes.data, n_expert,
                                     expert_stride, ids.ctypes.data, k, in_dim, out_dim,
                                     np.ascontiguousarray(xq).ctypes.data, int(x_per_pair), n_tok,
                                     pair.ctypes.data, row.ctypes.data, pair.size)
        if rc < 0:
            raise ValueError("oracle moe_sample: bad arguments")
        return out, bound, rc

    # -- the expert FFN around the routed product ----------------------------------
    def swiglu(self, gate, up, limit: float):
        """mid = silu(gate') * up' (gate' = min(gate, limit), up' = up clamped to
        [-limit, limit]; limit = 0: no clamp), float32, same shape as gate."""
        gate = np.ascontiguousarray(gate, dtype=np.float32)
        up = np.ascontiguousarray(up, dtype=np.float32)
        assert gate.shape == up.shape
        mid = np.empty_like(gate)
        self.lib.q8o_swiglu(mid.ctypes.data, gate.ctypes.data, up.ctypes.data, gate.size, float(limit))
        return mid

    def combine(self, y, w, n_tok: int, k: int):
        """y float32 [n_tok*k, dim], w float32 [n_tok*k] -> (out float64 [n_tok, dim], bound)."""
        y = np.ascontiguousarray(y, dtype=np.float32)
        w = np.ascontiguousarray(w, dtype=np.float32).reshape(-1)
        dim = y.shape[1]
        assert y.shape[0] == n_tok * k and w.size == n_tok * k
        out = np.empty((n_tok, dim), dtype=np.float64)
        bound = np.empty((n_tok, dim), dtype=np.float64)
        self.lib.q8o_combine(out.ctypes.data, bound.ctypes.data, y.ctypes.data, w.ctypes.data, n_tok, k, dim)
        return out, bound

    def moe_ffn(self, W_gate, W_up, W_down, n_expert, gate_up_stride, down_stride, ids, w, in_dim, mid_dim,
                out_dim, limit, x):
        """The routed expert FFN.  x float32 [n_tok, in_dim]; ids int32 and w float32 [n_tok, k].
        Returns a dict: out (float64 [n_tok, out_dim]), out_bound, y (float32 [n_tok*k, out_dim]),
        y_bound, mid (float32 [n_tok*k, mid_dim]), midq (its blocks), flag."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        n_tok = x.shape[0]
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        w = np.ascontiguousarray(w, dtype=np.float32)
        k = ids.size // n_tok if n_tok else 1
        n_pairs = n_tok * k
        r = {"out": np.empty((n_tok, out_dim), np.float64), "out_bound": np.empty((n_tok, out_dim), np.float64),
             "y": np.empty((n_pairs, out_dim), np.float32), "y_bound": np.empty((n_pairs, out_dim), np.float64),
             "mid": np.empty((n_pairs, mid_dim), np.float32),
             "midq": np.empty((n_pairs, mid_dim // QK * QBYTES), np.uint8)}
        rc = self.lib.q8o_moe_ffn(r["out"].ctypes.data, r["out_bound"].ctypes.data, r["y"].ctypes.data,
                                  r["y_bound"].ctypes.data, r["mid"].ctypes.data, r["midq"].ctypes.data,
                                  np.ascontiguousarray(W_gate).ctypes.data, np.ascontiguousarray(W_up).ctypes.data,
                                  np.ascontiguousarray(W_down).ctypes.data, n_expert, gate_up_stride, down_stride,
                                  ids.ctypes.data, w.ctypes.data, k, in_dim, mid_dim, out_dim, float(limit),
                                  x.ctypes.data, n_tok)
        if rc < 0:
            raise ValueError("oracle moe_ffn: bad dimensions")
        r["flag"] = rc
        return r

    # -- RMSNorm feeding the quantiser ----------------------------------------------
    def rmsnorm_quantize(self, x, gamma, eps: float):
        """x float32 [n_tok, dim], gamma float32 [dim] or None -> (xq uint8 [n_tok, dim/32*34],
        y float32 [n_tok, dim])."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        n_tok, dim = x.shape
        g = None if gamma is None else np.ascontiguousarray(gamma, dtype=np.float32)
        y = np.empty_like(x)
        xq = np.empty((n_tok, dim // QK * QBYTES), dtype=np.uint8)
        rc = self.lib.q8o_rmsnorm_quantize(xq.ctypes.data, y.ctypes.data, x.ctypes.data,
                                           None if g is None else g.ctypes.data, dim, n_tok, float(eps))
        if rc != 0:
            raise ValueError("oracle rmsnorm_quantize: bad dims")
        return xq, y

    # -- second weight format: Q2_K / Q4_K super-blocks against Q8_K activations -----
    def kq_block_bytes(self, fmt: int) -> int:
        return int(self.lib.q8o_kq_block_bytes(int(fmt)))

    def kq_dequant(self, W: np.ndarray, fmt: int, in_dim: int, rows: int) -> np.ndarray:
        """Raw K-quant rows -> float64 [rows, in_dim] weight values."""
        W = np.ascontiguousarray(W, dtype=np.uint8)
        assert W.nbytes == rows * in_dim // QKK * self.kq_block_bytes(fmt)
        out = np.empty((rows, in_dim), dtype=np.float64)
        if self.lib.q8o_kq_dequant(out.ctypes.data, W.ctypes.data, int(fmt), in_dim, rows) != 0:
            raise ValueError("oracle kq_dequant: bad format or dims")
        return out

    def quantize_q8k(self, x: np.ndarray):
        """x float32 [n_tok, in_dim] -> (d float32 [n_tok, in_dim/256], q int8 [n_tok, in_dim])."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim == 1:
            x = x[None, :]
        n_tok, in_dim = x.shape
        d = np.empty((n_tok, in_dim // QKK), dtype=np.float32)
        q = np.empty((n_tok, in_dim), dtype=np.int8)
        if self.lib.q8o_quantize_q8k(d.ctypes.data, q.ctypes.data, x.ctypes.data, in_dim, n_tok) != 0:
            raise ValueError("oracle quantize_q8k: bad dims")
        return d, q

    def kq_matmul_q(self, W, fmt: int, in_dim: int, out_dim: int, dx, qx):
        """K-quant rows W [out_dim] against Q8_K rows (dx [n_tok, in_dim/256], qx [n_tok, in_dim]).
        Returns (out float32 [n_tok, out_dim], bound float64 [n_tok, out_dim])."""
        dx = np.ascontiguousarray(dx, dtype=np.float32)
        qx = np.ascontiguousarray(qx, dtype=np.int8)
        n_tok = qx.shape[0]
        W = np.ascontiguousarray(W, dtype=np.uint8)
        assert W.nbytes == out_dim * in_dim // QKK * self.kq_block_bytes(fmt) and qx.shape[1] == in_dim
        out = np.empty((n_tok, out_dim), dtype=np.float32)
        bound = np.empty((n_tok, out_dim), dtype=np.float64)
        if self.lib.q8o_kq_matmul_q(out.ctypes.data, bound.ctypes.data, W.ctypes.data, int(fmt), in_dim, out_dim,
                                    dx.ctypes.data, qx.ctypes.data, n_tok) != 0:
            raise ValueError("oracle kq_matmul: bad format or dims")
        return out, bound

    def kq_matmul(self, W, fmt: int, x, out_dim: int):
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim == 1:
            x = x[None, :]
        dx, qx = self.quantize_q8k(x)
        return self.kq_matmul_q(W, fmt, x.shape[1], out_dim, dx, qx)

    def kq_moe(self, W_experts, fmt: int, n_expert: int, expert_stride: int, ids, in_dim: int, out_dim: int, x,
               x_per_pair: int):
        """Routed K-quant experts; x float32 [n_tok or n_tok*k, in_dim] is quantised to Q8_K here.
        Returns (out [n_tok*k, out_dim], bound, flag)."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        n_tok, k = ids.shape
        dx, qx = self.quantize_q8k(x)
        out = np.empty((n_tok * k, out_dim), dtype=np.float32)
        bound = np.empty((n_tok * k, out_dim), dtype=np.float64)
        rc = self.lib.q8o_kq_moe(out.ctypes.data, bound.ctypes.data, np.ascontiguousarray(W_experts).ctypes.data,
                                 int(fmt), n_expert, expert_stride, ids.ctypes.data, k, in_dim, out_dim,
                                 dx.ctypes.data, qx.ctypes.data, int(x_per_pair), n_tok)
        if rc < 0:
            raise ValueError("oracle kq_moe: bad dims")
        return out, bound, rc


_oracle = None


def get() -> Oracle:
    """The oracle built from q8_oracle.c (compiled on first use)."""
    global _oracle
    with _lock:
        if _oracle is None:
            _oracle = Oracle(build())
    return _oracle


def tolerance(bound: np.ndarray) -> np.ndarray:
    """Allowed |gpu - oracle| per output: 1e-4 * sum_b |d_w d_x isum_b| + 1e-6."""
    return 1e-4 * bound + 1e-6


def _deq_abs(raw, nb):
    """|d q| of raw Q8_0 rows [rows, nb*34] as float64 [rows, nb*32]."""
    r = raw.reshape(raw.shape[0], nb, QBYTES)
    d = (r[..., 0].astype(np.uint16) | (r[..., 1].astype(np.uint16) << 8)).view(np.float16).astype(np.float64)
    q = r[..., 2:].copy().view(np.int8).astype(np.float64)
    return np.abs(d[..., None] * q).reshape(raw.shape[0], nb * QK)


def ffn_tolerance(r, W_down, down_stride, ids, w, mid_dim, out_dim):
    """Allowed |gpu - oracle| per output of the routed expert FFN, from the oracle's result r
    (Oracle.moe_ffn).  Per pair: the matmul bound 1e-4 B + 1e-6 of the down projection
    (B = y_bound); 2^-10 B for a block whose binary16 scale rounds the other way; one
    quantisation step for every mid value whose quotient mid/d (d = amax/127 in fp32) lies
    within 1e-3 of a rounding tie, where fp32 differences in gate and up can flip its code;
    all weighted by |w|.  Then 2k 2^-24 sum_j |w_j y_j| for the fp32 weighted sum.  Pairs
    whose id is out of range have zero mid and y on both sides; pass any valid id for them."""
    ids = np.asarray(ids)
    n_tok, k = ids.shape
    nbm = mid_dim // QK
    blk = r["mid"].reshape(-1, nbm, QK)
    d = np.abs(blk).max(-1).astype(np.float32) / np.float32(127.0)
    with np.errstate(divide="ignore", invalid="ignore"):
        quo = np.abs(blk / d[..., None])
    risk = (np.abs(quo - np.floor(quo) - 0.5) < 1e-3) & (d[..., None] > 0)
    mq = r["midq"].reshape(-1, nbm, QBYTES)
    dh = (mq[..., 0].astype(np.uint16) | (mq[..., 1].astype(np.uint16) << 8)).view(np.float16).astype(np.float64)
    step = (risk * dh[..., None]).reshape(-1, mid_dim)
    tol = 2 * k * 2.0 ** -24 * r["out_bound"]
    row_bytes = nbm * QBYTES
    W_down = np.asarray(W_down).reshape(-1)
    for t in range(n_tok):
        for j in range(k):
            p, e = t * k + j, int(ids[t, j])
            flips = 0.0
            if step[p].any():
                We = W_down[e * down_stride:e * down_stride + out_dim * row_bytes].reshape(out_dim, row_bytes)
                flips = _deq_abs(We, nbm) @ step[p]
            tol[t] += abs(float(w[t, j])) * ((1e-4 + 2.0 ** -10) * r["y_bound"][p] + 1e-6 + flips)
    return tol
