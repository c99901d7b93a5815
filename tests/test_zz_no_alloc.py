"""q8_matmul_noalloc: the matmul for callers that must not allocate device memory
through this library (an application whose own pool allocator owns the device's
memory, or a decode loop that cannot take a first-use cudaMalloc).  Its output
must match q8_matmul's on the same inputs, within the parity tolerance, on two
calls in a row.  Collected last (file name) so that a run stopping at the first
failure has already run every other test; it also passes on its own."""
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


def test_noalloc_matches_q8_matmul_on_two_calls(q8):
    o = oracle.get()
    cases = [(1024, 4096, 4, 101), (4096, 1024, 16, 102)]   # two calls in a row, different shapes
    for in_dim, out_dim, n_tok, seed in cases:
        Wh = inputs.weights(out_dim, in_dim, seed=seed)
        xh = inputs.normal((n_tok, in_dim), seed=seed + 1, p_out=0.01)
        W = torch.from_numpy(Wh).cuda()
        x = torch.from_numpy(xh).cuda()
        ref = torch.empty((n_tok, out_dim), device="cuda")
        got = torch.full((n_tok, out_dim), float("nan"), device="cuda")
        assert q8.lib.q8_matmul(ref.data_ptr(), W.data_ptr(), in_dim, out_dim, x.data_ptr(), n_tok,
                                torch.cuda.current_stream().cuda_stream) == 0
        rc = q8.lib.q8_matmul_noalloc(got.data_ptr(), W.data_ptr(), in_dim, out_dim, x.data_ptr(), n_tok,
                                      torch.cuda.current_stream().cuda_stream)
        assert rc == 0, q8.q8_strerror(rc)
        assert q8.q8_last_error() == 0
        _, bound = o.matmul(Wh, xh, out_dim)
        g, r = got.cpu().numpy(), ref.cpu().numpy()
        assert not np.any(np.isnan(g))
        assert np.all(np.abs(g.astype(np.float64) - r) <= oracle.tolerance(bound))


def test_noalloc_rejects_calls_beyond_its_scratch(q8):
    # n_tok 512 x in_dim 32768 needs ~18 MiB of planes: refused before anything is enqueued.
    A = 0x10000
    rc = q8.lib.q8_matmul_noalloc(A, A, 32768, 1024, A, 512, None)
    assert rc == q8.Q8_ESCRATCH
    assert "fixed scratch" in q8.q8_strerror(rc)
