"""q8_matmul_noalloc: the matmul for callers that must not allocate device memory
through this library (an application whose own pool allocator owns the device's
memory, or a decode loop that cannot take a first-use cudaMalloc).

Its outputs are checked against the CPU oracle's exact values and against
q8_matmul's outputs on the same inputs, within the parity tolerance, on calls
in a row, for every kernel it can run: the GEMV from activation planes (up to
16 tokens), the mma.sync kernel (more tokens) and the plain kernel (rows that
are not 16-byte aligned).  Collected last (file name) so that a run stopping at
the first failure has already run every other test; it also passes on its own.
"""
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


def _check_calls(q8, cases):
    """Each case runs q8_matmul, then q8_matmul_noalloc, on one stream; the cases run
    back to back, so consecutive no-alloc calls reuse the fixed array."""
    o = oracle.get()
    st = torch.cuda.current_stream().cuda_stream
    for in_dim, out_dim, n_tok, seed in cases:
        Wh = inputs.weights(out_dim, in_dim, seed=seed)
        xh = inputs.normal((n_tok, in_dim), seed=seed + 1, p_out=0.01)
        W = torch.from_numpy(Wh).cuda()
        x = torch.from_numpy(xh).cuda()
        ref = torch.empty((n_tok, out_dim), device="cuda")
        got = torch.full((n_tok, out_dim), float("nan"), device="cuda")
        assert q8.lib.q8_matmul(ref.data_ptr(), W.data_ptr(), in_dim, out_dim, x.data_ptr(), n_tok, st) == 0
        rc = q8.lib.q8_matmul_noalloc(got.data_ptr(), W.data_ptr(), in_dim, out_dim, x.data_ptr(), n_tok, st)
        assert rc == 0, f"{q8.q8_strerror(rc)} {q8.q8_last_cuda_error()}"
        assert q8.q8_last_error() == 0
        exact, bound = o.matmul(Wh, xh, out_dim)
        tol = oracle.tolerance(bound)
        g, r = got.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)
        what = f"in {in_dim} out {out_dim} n_tok {n_tok}"
        assert not np.any(np.isnan(g)), f"{what}: output not written"
        assert np.all(np.abs(g - exact) <= tol), f"{what}: differs from the oracle"
        assert np.all(np.abs(g - r) <= tol), f"{what}: differs from q8_matmul"


def test_noalloc_matches_q8_matmul_on_two_calls(q8):
    # the weight-streaming GEMV, two calls in a row of different shapes
    _check_calls(q8, [(1024, 4096, 4, 101), (4096, 1024, 16, 102)])


def test_noalloc_other_kernels(q8):
    _check_calls(q8, [
        (4096, 1024, 64, 103),    # more than 16 tokens: the mma.sync kernel
        (1024, 300, 40, 104),     # ... with a ragged last row tile and token tile
        (1088, 70, 20, 105),      # in_dim / 32 = 34, even but not a multiple of 8: the plain kernel
        (96, 19, 7, 106),         # three blocks a row: the plain kernel
        (1024, 300, 40, 104),     # the first shape again after the others
    ])


def test_noalloc_rejects_calls_beyond_its_scratch(q8):
    # n_tok 512 x in_dim 32768 needs ~18 MiB of planes: refused before anything is enqueued.
    A = 0x10000
    rc = q8.lib.q8_matmul_noalloc(A, A, 32768, 1024, A, 512, None)
    assert rc == q8.Q8_ESCRATCH
    assert "fixed scratch" in q8.q8_strerror(rc)
