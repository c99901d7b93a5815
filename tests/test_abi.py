"""The C-ABI library loads and exports every symbol include/q8.h declares, and
its host-side validation rejects bad arguments before touching a GPU (no GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def q8():
    from q8_quantized_matmul_gb300 import build
    build.build()
    import q8_quantized_matmul_gb300 as m
    return m


def declared_functions():
    with open(os.path.join(ROOT, "include", "q8.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q8_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("q8_quantize_act", "q8_matmul", "q8_moe_matmul"):
        assert n in names


def test_library_exports_every_declared_symbol(q8):
    lib = ctypes.CDLL(q8.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/q8.h but not exported"
    assert set(declared_functions()) == set(q8.EXPORTS)


def test_version_and_strerror(q8):
    assert q8.q8_version() >= 10000
    assert q8.q8_strerror(q8.Q8_ERANGE) == "expert id out of range"
    assert q8.q8_strerror(12345) == "unknown status"


def test_repack_bytes_per_layout(q8):
    # split planes: the same 34 bytes per 32 weights
    assert q8.q8_repack_bytes(4096, 1024, q8.Q8_LAYOUT_PLANES) == 1024 * 128 * 34
    assert q8.q8_repack_bytes(33, 10, q8.Q8_LAYOUT_PLANES) == 0
    # tensor-core operand: fp16 quants and fp32 block-major scales over rows rounded up to 128
    assert q8.q8_repack_bytes(4096, 1000, q8.Q8_LAYOUT_TC) == 1024 * 4096 * 2 + 128 * 1024 * 4
    assert q8.q8_repack_bytes(96, 10, q8.Q8_LAYOUT_TC) == 0          # in_dim not a multiple of 64
    assert q8.q8_repack_bytes(4096, 1024, 2) == 0                     # unknown layout


def test_repack_rejects_bad_layouts_before_any_launch(q8):
    A = 0x10000
    assert q8.lib.q8_repack(A, A, 4096, 16, 7, None) == q8.Q8_EINVAL
    assert q8.lib.q8_repack(A, A, 96, 16, q8.Q8_LAYOUT_TC, None) == q8.Q8_EINVAL
    assert q8.lib.q8_matmul_packed(A, A, 3, 4096, 16, A, 1, None) == q8.Q8_EINVAL
    assert q8.lib.q8_matmul_packed(A, A, q8.Q8_LAYOUT_TC, 96, 16, A, 1, None) == q8.Q8_EINVAL


# Host validation: fake (never dereferenced) addresses, returns before any CUDA call.
A = 0x10000  # 16-byte aligned fake address
B = 0x20000


@pytest.mark.parametrize("in_dim", [0, 31, 33, 48])
def test_bad_in_dim_rejected(q8, in_dim):
    assert q8.lib.q8_matmul(A, B, in_dim, 8, A, 1, None) == q8.Q8_EINVAL
    assert q8.lib.q8_quantize_act(A, B, in_dim, 1, None) == q8.Q8_EINVAL
    assert q8.lib.q8_moe_matmul(A, B, 4, 1 << 20, A, 2, in_dim, 8, A, 0, 3, None) == q8.Q8_EINVAL


def test_null_and_misaligned_pointers_rejected(q8):
    assert q8.lib.q8_matmul(0, B, 64, 8, A, 1, None) == q8.Q8_EINVAL
    assert q8.lib.q8_matmul(A, 0, 64, 8, A, 1, None) == q8.Q8_EINVAL
    assert q8.lib.q8_matmul(A + 4, B, 64, 8, A, 1, None) == q8.Q8_EALIGN
    assert q8.lib.q8_matmul(A, B + 2, 64, 8, A, 1, None) == q8.Q8_EALIGN
    assert q8.lib.q8_matmul_q(A, B, 64, 8, A + 8, 1, None) == q8.Q8_EALIGN
    assert q8.lib.q8_quantize_act(A + 1, B, 64, 1, None) == q8.Q8_EALIGN


def test_moe_argument_checks(q8):
    L = q8.lib
    stride = 8 * 2 * 34  # out 8, in 64 -> 8 rows x 2 blocks
    assert L.q8_moe_matmul(A, B, 0, stride, A, 1, 64, 8, A, 0, 1, None) == q8.Q8_EINVAL       # no experts
    assert L.q8_moe_matmul(A, B, 4, stride, A, 5, 64, 8, A, 0, 1, None) == q8.Q8_EINVAL       # k > n_expert
    assert L.q8_moe_matmul(A, B, 4, stride - 16, A, 2, 64, 8, A, 0, 1, None) == q8.Q8_EINVAL  # stride too small
    assert L.q8_moe_matmul(A, B, 4, stride + 8, A, 2, 64, 8, A, 0, 1, None) == q8.Q8_EALIGN   # stride % 16
    assert L.q8_moe_matmul(A, B, 4, stride, A + 2, 2, 64, 8, A, 0, 1, None) == q8.Q8_EALIGN   # ids % 4
    assert L.q8_moe_matmul(A, B, 1 << 20, stride, A, 2, 64, 8, A, 0, 1, None) == q8.Q8_EINVAL  # too many experts


def test_empty_work_is_a_no_op(q8):
    # n_tok == 0 or out_dim == 0 returns before touching the device
    assert q8.lib.q8_matmul(A, B, 64, 8, A, 0, None) == q8.Q8_OK
    assert q8.lib.q8_matmul(A, B, 64, 0, A, 5, None) == q8.Q8_OK
    assert q8.lib.q8_quantize_act(A, B, 64, 0, None) == q8.Q8_OK


def test_overflowing_sizes_rejected(q8):
    assert q8.lib.q8_matmul(A, B, 1 << 32, 8, A, 1, None) == q8.Q8_EINVAL
    assert q8.lib.q8_matmul(A, B, 64, 1 << 40, A, 1, None) == q8.Q8_EINVAL


def test_no_gpu_means_error_not_crash(q8):
    """Without a usable sm_103a device the first real call reports Q8_ECUDA."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert q8.lib.q8_matmul(A, B, 64, 8, A, 1, None) == q8.Q8_ECUDA


def _no_gpu():
    import torch
    return not torch.cuda.is_available()


def test_matmul_host_argument_checks(q8):
    L = q8.lib
    assert L.q8_matmul_host(A, B, 64, 8, 0, 1, None) == q8.Q8_EINVAL        # no host x
    assert L.q8_matmul_host(0, B, 64, 8, A, 1, None) == q8.Q8_EINVAL        # no host out
    assert L.q8_matmul_host(A, B + 8, 64, 8, A, 1, None) == q8.Q8_EALIGN    # device W misaligned
    assert L.q8_matmul_host(A, B, 48, 8, A, 1, None) == q8.Q8_EINVAL
    assert L.q8_matmul_host(A, B, 64, 8, A, 0, None) == q8.Q8_OK
    if _no_gpu():   # host buffers need no alignment: these pass validation and reach the device check
        assert L.q8_matmul_host(A + 4, B, 64, 8, A + 3, 1, None) == q8.Q8_ECUDA


def test_moe_ffn_argument_checks(q8):
    L = q8.lib
    gu, ds = 32 * 2 * 34, 16 * 1 * 34 + 8   # gate/up: mid 32 rows x 2 blocks; down: 16 rows x 1 block (+8)
    ds16 = ds + 8

    def call(**kw):
        a = dict(out=A, Wg=B, Wu=B, Wd=B, n_exp=4, gu=gu, ds=ds16, ids=A, w=A, k=2, in_dim=64, mid=32, out_dim=16,
                 limit=10.0, x=A, n_tok=3)
        a.update(kw)
        return L.q8_moe_ffn(a["out"], a["Wg"], a["Wu"], a["Wd"], a["n_exp"], a["gu"], a["ds"], a["ids"], a["w"],
                            a["k"], a["in_dim"], a["mid"], a["out_dim"], a["limit"], a["x"], a["n_tok"], None)
    assert call(limit=float("nan")) == q8.Q8_EINVAL
    assert call(limit=-1.0) == q8.Q8_EINVAL
    assert call(mid=48) == q8.Q8_EINVAL                 # mid_dim % 32
    assert call(k=5) == q8.Q8_EINVAL                    # k > n_expert
    assert call(gu=gu - 16) == q8.Q8_EINVAL             # gate/up stride shorter than a matrix
    assert call(ds=16 * 34 - 16) == q8.Q8_EINVAL        # down stride shorter than a matrix
    assert call(ds=ds) == q8.Q8_EALIGN                  # down stride not a multiple of 16
    assert call(ids=A + 2) == q8.Q8_EALIGN
    assert call(w=A + 2) == q8.Q8_EALIGN
    assert call(x=A + 4) == q8.Q8_EALIGN
    assert call(w=0) == q8.Q8_EINVAL
    assert call(n_tok=0) == q8.Q8_OK
    if _no_gpu():
        assert call() == q8.Q8_ECUDA


def test_elementwise_and_norm_argument_checks(q8):
    L = q8.lib
    assert L.q8_swiglu(A, A, A, 8, float("nan"), None) == q8.Q8_EINVAL
    assert L.q8_swiglu(A, A, A, 8, -0.5, None) == q8.Q8_EINVAL
    assert L.q8_swiglu(A, A, A, 0, 1.0, None) == q8.Q8_OK
    assert L.q8_swiglu(0, A, A, 8, 1.0, None) == q8.Q8_EINVAL
    assert L.q8_swiglu(A, A + 4, A, 8, 1.0, None) == q8.Q8_EALIGN
    assert L.q8_moe_combine(A, A, A, 2, 0, 8, None) == q8.Q8_EINVAL        # k = 0
    assert L.q8_moe_combine(A, A, A, 0, 2, 8, None) == q8.Q8_OK
    assert L.q8_moe_combine(A, 0, A, 2, 2, 8, None) == q8.Q8_EINVAL
    assert L.q8_moe_combine(A + 4, A, A, 2, 2, 8, None) == q8.Q8_EALIGN
    assert L.q8_moe_combine(A, A, A + 2, 2, 2, 8, None) == q8.Q8_EALIGN
    for eps in (0.0, -1.0, float("nan"), float("inf")):
        assert L.q8_rmsnorm_quantize(A, 0, B, 0, 64, 2, eps, None) == q8.Q8_EINVAL
    assert L.q8_rmsnorm_quantize(A, 0, B, 0, 48, 2, 1e-6, None) == q8.Q8_EINVAL
    assert L.q8_rmsnorm_quantize(0, 0, B, 0, 64, 2, 1e-6, None) == q8.Q8_EINVAL
    assert L.q8_rmsnorm_quantize(A, A + 4, B, 0, 64, 2, 1e-6, None) == q8.Q8_EALIGN   # y misaligned
    assert L.q8_rmsnorm_quantize(A, 0, B, B + 8, 64, 2, 1e-6, None) == q8.Q8_EALIGN   # gamma misaligned
    assert L.q8_rmsnorm_quantize(A, 0, B, 0, 64, 0, 1e-6, None) == q8.Q8_OK
    if _no_gpu():
        assert L.q8_swiglu(A, A, A, 8, 1.0, None) == q8.Q8_ECUDA
        assert L.q8_moe_combine(A, A, A, 2, 2, 8, None) == q8.Q8_ECUDA
        assert L.q8_rmsnorm_quantize(A, 0, B, 0, 64, 2, 1e-6, None) == q8.Q8_ECUDA


def test_kquant_argument_checks(q8):
    """The second weight format's entry points: bad formats, dimensions, strides and alignments are
    rejected on the host; empty work is a no-op."""
    L = q8.lib
    assert q8.q8_kq_row_bytes(512, q8.Q8_KQ_Q2_K) == 2 * 84 and q8.q8_kq_row_bytes(512, q8.Q8_KQ_Q4_K) == 2 * 144
    assert q8.q8_kq_row_bytes(512, 3) == 0 and q8.q8_kq_row_bytes(320, q8.Q8_KQ_Q4_K) == 0
    for fmt in (0, 3, 8):
        assert L.q8_kq_matmul(A, B, fmt, 512, 8, A, 1, None) == q8.Q8_EINVAL
    for in_dim in (0, 32, 128, 320):
        assert L.q8_kq_matmul(A, B, q8.Q8_KQ_Q4_K, in_dim, 8, A, 1, None) == q8.Q8_EINVAL
        assert L.q8_quantize_q8k(A, B, in_dim, 1, None) == q8.Q8_EINVAL
    assert L.q8_kq_matmul(A, B + 4, q8.Q8_KQ_Q4_K, 512, 8, A, 1, None) == q8.Q8_EALIGN   # Q4_K rows: 16 bytes
    assert L.q8_kq_matmul(A, B + 2, q8.Q8_KQ_Q2_K, 512, 8, A, 1, None) == q8.Q8_EALIGN   # Q2_K rows: 4 bytes
    assert L.q8_kq_matmul(A, B, q8.Q8_KQ_Q4_K, 512, 8, A + 8, 1, None) == q8.Q8_EALIGN   # x
    assert L.q8_quantize_q8k(A + 2, B, 512, 1, None) == q8.Q8_EALIGN
    assert L.q8_kq_matmul(A, B, q8.Q8_KQ_Q4_K, 512, 8, A, 0, None) == q8.Q8_OK
    assert L.q8_kq_matmul(A, B, q8.Q8_KQ_Q4_K, 512, 0, A, 3, None) == q8.Q8_OK
    assert L.q8_quantize_q8k(A, B, 512, 0, None) == q8.Q8_OK
    stride = 8 * 2 * 144
    m = L.q8_kq_moe_matmul
    assert m(A, B, q8.Q8_KQ_Q4_K, 0, stride, A, 1, 512, 8, A, 0, 1, None) == q8.Q8_EINVAL       # no experts
    assert m(A, B, q8.Q8_KQ_Q4_K, 4, stride, A, 5, 512, 8, A, 0, 1, None) == q8.Q8_EINVAL       # k > n_expert
    assert m(A, B, q8.Q8_KQ_Q4_K, 4, stride - 16, A, 2, 512, 8, A, 0, 1, None) == q8.Q8_EINVAL  # stride too small
    assert m(A, B, q8.Q8_KQ_Q4_K, 4, stride + 4, A, 2, 512, 8, A, 0, 1, None) == q8.Q8_EALIGN   # stride % 16
    assert m(A, B, q8.Q8_KQ_Q2_K, 4, 8 * 2 * 84 + 2, A, 2, 512, 8, A, 0, 1, None) == q8.Q8_EALIGN   # stride % 4
    assert m(A, B, q8.Q8_KQ_Q4_K, 4, stride, A + 2, 2, 512, 8, A, 0, 1, None) == q8.Q8_EALIGN   # ids
    assert m(A, B, q8.Q8_KQ_Q4_K, 4, stride, A, 2, 512, 8, A, 0, 0, None) == q8.Q8_OK
    if _no_gpu():
        assert L.q8_kq_matmul(A, B, q8.Q8_KQ_Q2_K, 512, 8, A, 1, None) == q8.Q8_ECUDA
        assert m(A, B, q8.Q8_KQ_Q4_K, 4, stride, A, 2, 512, 8, A, 0, 1, None) == q8.Q8_ECUDA
