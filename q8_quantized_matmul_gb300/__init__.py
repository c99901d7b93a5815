"""Thin Python binding of the GB300 Q8_0 x Q8_0 matmul library (include/q8.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libq8.so``.  There is no CPU fallback: importing this package
fails loudly when the library is missing or cannot be loaded.

Functions keep the C names.  Tensors are PyTorch tensors on the current CUDA
device (PyTorch supplies device memory and streams); each call is enqueued on
``torch.cuda.current_stream()`` unless a stream is given, and returns the
C status code (0 = Q8_OK).  ``Q8Error`` is raised by the ``*_checked`` helpers.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libq8.so")

QK = 32
QB = 34
Q8_OK, Q8_EINVAL, Q8_EALIGN, Q8_ERANGE, Q8_ENOMEM, Q8_ECUDA, Q8_ETIMEOUT, Q8_ESCRATCH = 0, -1, -2, -3, -4, -5, -6, -7
Q8_NOALLOC_SCRATCH_BYTES = 4 << 20
Q8_LAYOUT_PLANES, Q8_LAYOUT_TC = 0, 1
Q8_KQ_Q2_K, Q8_KQ_Q4_K = 2, 4
Q8_Q8K_BLOCK_BYTES = 292

# Every symbol include/q8.h declares.
EXPORTS = ("q8_version", "q8_strerror", "q8_quantize_act", "q8_matmul", "q8_matmul_q", "q8_moe_matmul",
           "q8_repack_bytes", "q8_repack", "q8_matmul_packed", "q8_last_error", "q8_scratch_bytes",
           "q8_release", "q8_debug_fail_next_alloc", "q8_profile_arm", "q8_profile_used", "q8_profile_read",
           "q8_matmul_noalloc", "q8_last_cuda_error", "q8_matmul_host", "q8_moe_ffn", "q8_swiglu",
           "q8_moe_combine", "q8_rmsnorm_quantize", "q8_debug_expire_waits", "q8_kq_row_bytes",
           "q8_quantize_q8k", "q8_kq_matmul", "q8_kq_moe_matmul")


class Q8Error(RuntimeError):
    def __init__(self, status: int, what: str):
        detail = f" [{_get().q8_last_cuda_error().decode()}]" if status == Q8_ECUDA else ""
        super().__init__(f"{what}: {_get().q8_strerror(status).decode()} ({status}){detail}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m q8_quantized_matmul_gb300.build` "
                          "(nvcc, sm_103a); there is no fallback path")
    L = ctypes.CDLL(LIB_PATH)
    vp, u64, u32, i32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int
    sig = {
        "q8_version": ([], i32),
        "q8_strerror": ([i32], ctypes.c_char_p),
        "q8_quantize_act": ([vp, vp, u64, u64, vp], i32),
        "q8_matmul": ([vp, vp, u64, u64, vp, u64, vp], i32),
        "q8_matmul_q": ([vp, vp, u64, u64, vp, u64, vp], i32),
        "q8_matmul_host": ([vp, vp, u64, u64, vp, u64, vp], i32),
        "q8_moe_matmul": ([vp, vp, u32, u64, vp, u32, u64, u64, vp, i32, u64, vp], i32),
        "q8_moe_ffn": ([vp, vp, vp, vp, u32, u64, u64, vp, vp, u32, u64, u64, u64, ctypes.c_float, vp, u64, vp],
                       i32),
        "q8_swiglu": ([vp, vp, vp, u64, ctypes.c_float, vp], i32),
        "q8_rmsnorm_quantize": ([vp, vp, vp, vp, u64, u64, ctypes.c_float, vp], i32),
        "q8_moe_combine": ([vp, vp, vp, u64, u32, u64, vp], i32),
        "q8_repack_bytes": ([u64, u64, i32], u64),
        "q8_repack": ([vp, vp, u64, u64, i32, vp], i32),
        "q8_matmul_packed": ([vp, vp, i32, u64, u64, vp, u64, vp], i32),
        "q8_last_error": ([vp], i32),
        "q8_scratch_bytes": ([], u64),
        "q8_release": ([], None),
        "q8_debug_fail_next_alloc": ([i32], None),
        "q8_debug_expire_waits": ([i32, u64], None),
        "q8_profile_arm": ([u32], i32),
        "q8_profile_used": ([], u64),
        "q8_profile_read": ([u32, ctypes.POINTER(ctypes.c_float)], i32),
        "q8_matmul_noalloc": ([vp, vp, u64, u64, vp, u64, vp], i32),
        "q8_last_cuda_error": ([], ctypes.c_char_p),
        "q8_kq_row_bytes": ([u64, i32], u64),
        "q8_quantize_q8k": ([vp, vp, u64, u64, vp], i32),
        "q8_kq_matmul": ([vp, vp, i32, u64, u64, vp, u64, vp], i32),
        "q8_kq_moe_matmul": ([vp, vp, i32, u32, u64, vp, u32, u64, u64, vp, i32, u64, vp], i32),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    return L


_lib = None


def _get() -> ctypes.CDLL:
    """The loaded library (loaded on first use; raises ImportError when it is missing)."""
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def __getattr__(name):
    if name == "lib":
        return _get()
    raise AttributeError(name)


def _p(t) -> int:
    """Device pointer of a tensor (or pass an int through)."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _s(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------------ same names as the C ABI
def q8_quantize_act(xq, x, in_dim: int, n_tok: int, stream=None) -> int:
    return _get().q8_quantize_act(_p(xq), _p(x), in_dim, n_tok, _s(stream))


def q8_matmul(out, W, in_dim: int, out_dim: int, x, n_tok: int, stream=None) -> int:
    return _get().q8_matmul(_p(out), _p(W), in_dim, out_dim, _p(x), n_tok, _s(stream))


def q8_matmul_noalloc(out, W, in_dim: int, out_dim: int, x, n_tok: int, stream=None) -> int:
    """q8_matmul with its scratch in the library's fixed device array (no allocation)."""
    return _get().q8_matmul_noalloc(_p(out), _p(W), in_dim, out_dim, _p(x), n_tok, _s(stream))


def q8_matmul_host(out_host, W, in_dim: int, out_dim: int, x_host, n_tok: int, stream=None) -> int:
    """q8_matmul with x and out in host memory (CPU tensors, ideally pinned); W on the device."""
    return _get().q8_matmul_host(_p(out_host), _p(W), in_dim, out_dim, _p(x_host), n_tok, _s(stream))


def q8_matmul_q(out, W, in_dim: int, out_dim: int, xq, n_tok: int, stream=None) -> int:
    return _get().q8_matmul_q(_p(out), _p(W), in_dim, out_dim, _p(xq), n_tok, _s(stream))


def q8_moe_matmul(out, W_experts, n_expert: int, expert_stride_bytes: int, expert_ids, k: int, in_dim: int,
                  out_dim: int, x, x_per_pair: int, n_tok: int, stream=None) -> int:
    return _get().q8_moe_matmul(_p(out), _p(W_experts), n_expert, expert_stride_bytes, _p(expert_ids), k, in_dim,
                             out_dim, _p(x), int(x_per_pair), n_tok, _s(stream))


def q8_moe_ffn(out, W_gate, W_up, W_down, n_expert: int, gate_up_stride_bytes: int, down_stride_bytes: int,
               expert_ids, expert_weights, k: int, in_dim: int, mid_dim: int, out_dim: int, limit: float, x,
               n_tok: int, stream=None) -> int:
    return _get().q8_moe_ffn(_p(out), _p(W_gate), _p(W_up), _p(W_down), n_expert, gate_up_stride_bytes,
                             down_stride_bytes, _p(expert_ids), _p(expert_weights), k, in_dim, mid_dim, out_dim,
                             float(limit), _p(x), n_tok, _s(stream))


def q8_rmsnorm_quantize(xq, y, x, gamma, dim: int, n_tok: int, eps: float, stream=None) -> int:
    return _get().q8_rmsnorm_quantize(_p(xq), _p(y), _p(x), _p(gamma), dim, n_tok, float(eps), _s(stream))


def q8_swiglu(mid, gate, up, n: int, limit: float, stream=None) -> int:
    return _get().q8_swiglu(_p(mid), _p(gate), _p(up), n, float(limit), _s(stream))


def q8_moe_combine(out, y, weights, n_tok: int, k: int, dim: int, stream=None) -> int:
    return _get().q8_moe_combine(_p(out), _p(y), _p(weights), n_tok, k, dim, _s(stream))


def q8_repack_bytes(in_dim: int, rows: int, layout: int = 0) -> int:
    return _get().q8_repack_bytes(in_dim, rows, layout)


def q8_repack(Wp, W, in_dim: int, rows: int, layout: int = 0, stream=None) -> int:
    return _get().q8_repack(_p(Wp), _p(W), in_dim, rows, layout, _s(stream))


def q8_matmul_packed(out, Wp, layout: int, in_dim: int, out_dim: int, x, n_tok: int, stream=None) -> int:
    return _get().q8_matmul_packed(_p(out), _p(Wp), layout, in_dim, out_dim, _p(x), n_tok, _s(stream))


def q8_kq_row_bytes(in_dim: int, fmt: int) -> int:
    return _get().q8_kq_row_bytes(in_dim, fmt)


def q8_quantize_q8k(xq, x, in_dim: int, n_tok: int, stream=None) -> int:
    return _get().q8_quantize_q8k(_p(xq), _p(x), in_dim, n_tok, _s(stream))


def q8_kq_matmul(out, W, fmt: int, in_dim: int, out_dim: int, x, n_tok: int, stream=None) -> int:
    return _get().q8_kq_matmul(_p(out), _p(W), fmt, in_dim, out_dim, _p(x), n_tok, _s(stream))


def q8_kq_moe_matmul(out, W_experts, fmt: int, n_expert: int, expert_stride_bytes: int, expert_ids, k: int,
                     in_dim: int, out_dim: int, x, x_per_pair: int, n_tok: int, stream=None) -> int:
    return _get().q8_kq_moe_matmul(_p(out), _p(W_experts), fmt, n_expert, expert_stride_bytes, _p(expert_ids), k,
                                   in_dim, out_dim, _p(x), x_per_pair, n_tok, _s(stream))


def q8_last_error(stream=None) -> int:
    return _get().q8_last_error(_s(stream))


def q8_scratch_bytes() -> int:
    return _get().q8_scratch_bytes()


def q8_release() -> None:
    _get().q8_release()


def q8_debug_fail_next_alloc(count: int) -> None:
    _get().q8_debug_fail_next_alloc(count)


def q8_debug_expire_waits(count: int, limit_ns: int) -> None:
    _get().q8_debug_expire_waits(count, limit_ns)


def q8_profile_arm(n_pairs: int) -> int:
    return _get().q8_profile_arm(n_pairs)


def q8_profile_used() -> int:
    return _get().q8_profile_used()


def q8_profile_read(i: int) -> float:
    """Elapsed milliseconds of timing pair i (raises if it was never recorded)."""
    ms = ctypes.c_float(0.0)
    _check(_get().q8_profile_read(i, ctypes.byref(ms)), "q8_profile_read")
    return ms.value


def q8_last_cuda_error() -> str:
    return _get().q8_last_cuda_error().decode()


def q8_strerror(status: int) -> str:
    return _get().q8_strerror(status).decode()


def q8_version() -> int:
    return _get().q8_version()


# ------------------------------------------------------------------ allocating helpers (torch)
def _check(rc: int, what: str) -> None:
    if rc != Q8_OK:
        raise Q8Error(rc, what)


def quantize_act(x):
    """x float32 [n_tok, in_dim] (cuda) -> uint8 [n_tok, in_dim/32*34] Q8_0 blocks."""
    import torch
    n_tok, in_dim = x.shape
    xq = torch.empty((n_tok, in_dim // QK * QB), dtype=torch.uint8, device=x.device)
    _check(q8_quantize_act(xq, x, in_dim, n_tok), "q8_quantize_act")
    return xq


def matmul(W, x, out_dim: int):
    """W uint8 raw Q8_0 rows [out_dim, in_dim/32*34]; x float32 [n_tok, in_dim] -> [n_tok, out_dim]."""
    import torch
    n_tok, in_dim = x.shape
    out = torch.empty((n_tok, out_dim), dtype=torch.float32, device=x.device)
    _check(q8_matmul(out, W, in_dim, out_dim, x, n_tok), "q8_matmul")
    return out


def matmul_q(W, xq, in_dim: int, out_dim: int):
    import torch
    n_tok = xq.shape[0]
    out = torch.empty((n_tok, out_dim), dtype=torch.float32, device=xq.device)
    _check(q8_matmul_q(out, W, in_dim, out_dim, xq, n_tok), "q8_matmul_q")
    return out


def moe_matmul(W_experts, n_expert: int, expert_stride: int, ids, x, x_per_pair: bool, out_dim: int):
    """ids int32 [n_tok, k]; x [n_tok, in] or [n_tok*k, in] -> [n_tok*k, out_dim]."""
    import torch
    n_tok, k = ids.shape
    in_dim = x.shape[1]
    out = torch.empty((n_tok * k, out_dim), dtype=torch.float32, device=x.device)
    _check(q8_moe_matmul(out, W_experts, n_expert, expert_stride, ids, k, in_dim, out_dim, x, int(x_per_pair),
                         n_tok), "q8_moe_matmul")
    return out


def moe_ffn(W_gate, W_up, W_down, n_expert: int, gate_up_stride: int, down_stride: int, ids, weights, x,
            mid_dim: int, out_dim: int, limit: float):
    """ids int32 and weights fp32 [n_tok, k]; x [n_tok, in] -> [n_tok, out_dim] (routed expert FFN)."""
    import torch
    n_tok, k = ids.shape
    in_dim = x.shape[1]
    out = torch.empty((n_tok, out_dim), dtype=torch.float32, device=x.device)
    _check(q8_moe_ffn(out, W_gate, W_up, W_down, n_expert, gate_up_stride, down_stride, ids, weights, k, in_dim,
                      mid_dim, out_dim, limit, x, n_tok), "q8_moe_ffn")
    return out


def rmsnorm_quantize(x, gamma, eps: float, want_y: bool = False):
    """x float32 [n_tok, dim] (cuda), gamma [dim] or None -> Q8_0 blocks [n_tok, dim/32*34]
    (and the normalised fp32 rows when want_y)."""
    import torch
    n_tok, dim = x.shape
    xq = torch.empty((n_tok, dim // QK * QB), dtype=torch.uint8, device=x.device)
    y = torch.empty_like(x) if want_y else None
    _check(q8_rmsnorm_quantize(xq, y, x, gamma, dim, n_tok, eps), "q8_rmsnorm_quantize")
    return (xq, y) if want_y else xq


def repack(W, in_dim: int, rows: int, layout: int = 0):
    import torch
    nbytes = q8_repack_bytes(in_dim, rows, layout)
    if nbytes == 0 and rows:
        raise Q8Error(Q8_EINVAL, "q8_repack_bytes")
    Wp = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    _check(q8_repack(Wp, W, in_dim, rows, layout), "q8_repack")
    return Wp


def matmul_packed(Wp, x, out_dim: int, layout: int = 0):
    import torch
    n_tok, in_dim = x.shape
    out = torch.empty((n_tok, out_dim), dtype=torch.float32, device=x.device)
    _check(q8_matmul_packed(out, Wp, layout, in_dim, out_dim, x, n_tok), "q8_matmul_packed")
    return out


def quantize_q8k(x):
    """x float32 [n_tok, in_dim] (cuda) -> uint8 [n_tok, in_dim/256*292] Q8_K blocks."""
    import torch
    n_tok, in_dim = x.shape
    xq = torch.empty((n_tok, in_dim // 256 * Q8_Q8K_BLOCK_BYTES), dtype=torch.uint8, device=x.device)
    _check(q8_quantize_q8k(xq, x, in_dim, n_tok), "q8_quantize_q8k")
    return xq


def kq_matmul(W, fmt: int, x, out_dim: int):
    """W uint8 K-quant rows [out_dim, q8_kq_row_bytes]; x float32 [n_tok, in_dim] -> [n_tok, out_dim]."""
    import torch
    n_tok, in_dim = x.shape
    out = torch.empty((n_tok, out_dim), dtype=torch.float32, device=x.device)
    _check(q8_kq_matmul(out, W, fmt, in_dim, out_dim, x, n_tok), "q8_kq_matmul")
    return out


def kq_moe_matmul(W_experts, fmt: int, n_expert: int, expert_stride: int, ids, x, x_per_pair: bool, out_dim: int):
    """ids int32 [n_tok, k]; x [n_tok, in] or [n_tok*k, in] -> [n_tok*k, out_dim] (K-quant experts)."""
    import torch
    n_tok, k = ids.shape
    in_dim = x.shape[1]
    out = torch.empty((n_tok * k, out_dim), dtype=torch.float32, device=x.device)
    _check(q8_kq_moe_matmul(out, W_experts, fmt, n_expert, expert_stride, ids, k, in_dim, out_dim, x,
                            int(x_per_pair), n_tok), "q8_kq_moe_matmul")
    return out
