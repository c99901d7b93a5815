"""Failure detection on the GPU without a fault: every wait inside the kernels is
bounded, and an expired wait ends the kernel with Q8_ETIMEOUT instead of a hang.

The test hook q8_debug_expire_waits makes the next dense kernel's producer issue
no copy at all (its consumers wait on buffers that never fill) and shortens the
wait limit.  The call must still return, the error word must read Q8_ETIMEOUT,
and the next call on the same context must pass oracle parity.  Covered: the
weight-streaming GEMV (fused quantiser, and behind the quantiser kernel) on the
decode projection shape, the tcgen05 GEMM on raw and on expanded weights, and
the TMA-fed RMSNorm kernel (its rows' copies withheld).
"""
import time

import numpy as np
import pytest

import inputs
import oracle

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def q8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from q8_quantized_matmul_gb300 import build
    build.build()
    import q8_quantized_matmul_gb300 as m
    torch.cuda.set_device(0)
    return m


LIMIT_NS = 200_000   # 0.2 ms instead of the normal 2 s


@pytest.mark.parametrize("in_dim,out_dim,n_tok", [
    (1024, 32768, 4),     # decode projection sweep shape: GEMV quantising in the kernel
    (1024, 32768, 16),    # ... behind the quantiser kernel
    (4096, 256, 64),      # prefill: tcgen05 GEMM on raw Q8_0 weights (K split over CTAs)
    (2112, 130, 700),     # tcgen05 GEMM on the expanded fp16 weights (two MMA issuers)
])
def test_expired_wait_reports_timeout_and_context_recovers(q8, in_dim, out_dim, n_tok):
    o = oracle.get()
    Wh = inputs.weights(out_dim, in_dim, seed=7)
    xh = inputs.normal((n_tok, in_dim), seed=8, p_out=0.01, out_scale=20.0)
    W, x = torch.from_numpy(Wh).cuda(), torch.from_numpy(xh).cuda()
    out = torch.full((n_tok, out_dim), float("nan"), device="cuda")
    assert q8.q8_last_error() == 0
    q8.q8_debug_expire_waits(1, LIMIT_NS)
    try:
        t0 = time.perf_counter()
        assert q8.q8_matmul(out, W, in_dim, out_dim, x, n_tok) == 0
        assert q8.q8_last_error() == q8.Q8_ETIMEOUT       # synchronises: the kernel ended
        assert time.perf_counter() - t0 < 1.5, "an expired wait did not end its kernel promptly"
    finally:
        q8.q8_debug_expire_waits(0, 0)
    assert q8.q8_last_error() == 0                        # read and cleared
    # the hook was used up by that one kernel: the next call is a normal one
    out.fill_(float("nan"))
    assert q8.q8_matmul(out, W, in_dim, out_dim, x, n_tok) == 0
    assert q8.q8_last_error() == 0
    ref, bound = o.matmul(Wh, xh, out_dim)
    got = out.cpu().numpy().astype(np.float64)
    assert not np.any(np.isnan(got))
    assert np.all(np.abs(got - ref) <= oracle.tolerance(bound))


def test_expired_wait_rmsnorm_tma(q8):
    """The TMA-fed RMSNorm kernel (rows of 4096 values, 12 rows per SM and more) issues no row copy
    under the hook: every CTA's waits expire, it skips its output and returns; the call ends promptly
    with Q8_ETIMEOUT and the next call on the context agrees with the oracle."""
    from tests import allowances
    o = oracle.get()
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    n_tok, dim = 12 * n_sm + 3, 4096
    xh = inputs.normal((n_tok, dim), seed=9, p_out=0.01)
    gh = (1.0 + 0.3 * np.random.default_rng(9).standard_normal(dim)).astype(np.float32)
    x, g = torch.from_numpy(xh).cuda(), torch.from_numpy(gh).cuda()
    assert q8.q8_last_error() == 0
    q8.q8_debug_expire_waits(1, LIMIT_NS)
    try:
        t0 = time.perf_counter()
        q8.rmsnorm_quantize(x, g, 1e-6, want_y=True)
        assert q8.q8_last_error() == q8.Q8_ETIMEOUT
        assert time.perf_counter() - t0 < 1.5, "an expired wait did not end its kernel promptly"
    finally:
        q8.q8_debug_expire_waits(0, 0)
    assert q8.q8_last_error() == 0
    xq, y = q8.rmsnorm_quantize(x, g, 1e-6, want_y=True)
    assert q8.q8_last_error() == 0
    xq_o, y_o = o.rmsnorm_quantize(xh, gh, 1e-6)
    allowances.check_rmsnorm(xq.cpu().numpy(), y.cpu().numpy(), xq_o, y_o)
