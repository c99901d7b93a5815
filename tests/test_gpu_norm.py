"""GPU parity of RMSNorm feeding the quantiser (q8_rmsnorm_quantize) through the C
ABI, against the CPU oracle.

* The quantised rows must be bit for bit the activation quantiser (q8_quantize_act,
  itself bit-exact to the oracle) applied to the kernel's own normalised rows y:
  the fused quantiser is the a1 quantiser.
* y and the quantised rows against the oracle's: the rules of tests/allowances.py
  (y within the relative bound of the kernel's fixed-order fp32 reduction; a quant
  or a binary16 scale one step apart only where that error can move the decision).
"""
import numpy as np
import pytest

import inputs
import oracle
from tests import allowances

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
QK, QB = 32, 34
DEV = "cuda:0"


@pytest.fixture(scope="module")
def q8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from q8_quantized_matmul_gb300 import build
    build.build()
    import q8_quantized_matmul_gb300 as m
    torch.cuda.set_device(0)
    return m


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def check(q8, o, x, gamma, eps):
    xq, y = q8.rmsnorm_quantize(dev(x), None if gamma is None else dev(gamma), eps, want_y=True)
    assert q8.q8_last_error() == 0
    # the fused quantiser is the activation quantiser of the kernel's own y
    assert torch.equal(xq, q8.quantize_act(y))
    xq_o, y_o = o.rmsnorm_quantize(x, gamma, eps)
    allowances.check_rmsnorm(xq.cpu().numpy(), y.cpu().numpy(), xq_o, y_o)
    return xq, y


@pytest.mark.parametrize("dim,n_tok", [(4096, 37), (1024, 5), (96, 3), (32, 7), (2080, 4), (6144, 9), (16384, 2),
                                       # more rows than resident CTAs: each CTA loops, the next row in flight
                                       (4096, 1000), (8192, 700), (2048, 2000),
                                       # 12 * 152 rows and more (rows <= 4096 values): the TMA-fed kernel,
                                       # one lane per block; 1, 3 and 65 blocks leave lanes of a warp idle
                                       (4096, 1900), (1024, 1824), (32, 2000), (96, 1900), (2080, 1830),
                                       # the long-prefill shape itself
                                       (4096, 4096)])
@pytest.mark.parametrize("with_gamma", [True, False])
def test_rmsnorm_quantize_parity(q8, o, dim, n_tok, with_gamma):
    x = inputs.normal((n_tok, dim), seed=dim + n_tok, p_out=0.01)
    g = np.random.default_rng(dim)
    gamma = (1.0 + 0.3 * g.standard_normal(dim)).astype(np.float32) if with_gamma else None
    check(q8, o, x, gamma, 1e-6)


def test_rmsnorm_quantize_many_rows_and_special_rows(q8, o):
    """More rows than resident CTAs (each CTA loops over rows), a zero row, a row where eps
    dominates, and a row of +/-1."""
    n_tok, dim = 152 * 8 + 5, 64
    check_special_rows(q8, o, n_tok, dim)


def test_rmsnorm_quantize_special_rows_tma(q8, o):
    """The same special rows through the TMA-fed kernel (enough rows for three per CTA)."""
    check_special_rows(q8, o, 152 * 12 + 7, 256)


def check_special_rows(q8, o, n_tok, dim):
    x = inputs.normal((n_tok, dim), seed=7)
    x[3] = 0.0
    x[10] = (1e-6 * x[10]).astype(np.float32)
    x[11] = np.where(np.arange(dim) % 3 == 0, -1.0, 1.0)
    gamma = (0.5 + np.random.default_rng(8).random(dim)).astype(np.float32)
    xq, y = check(q8, o, x, gamma, 1e-3)
    assert torch.all(y[3] == 0) and torch.all(xq[3] == 0)


def test_rmsnorm_quantize_deterministic_and_feeds_matmul(q8):
    """Same bits on every run; and the quantised rows feed q8_matmul_q with the result of
    q8_matmul on the normalised rows (the separate quantiser pass this kernel replaces)."""
    n_tok, dim, out_dim = 16, 4096, 1000
    x = dev(inputs.normal((n_tok, dim), seed=9, p_out=0.01))
    gamma = dev((1.0 + 0.1 * np.random.default_rng(10).standard_normal(dim)).astype(np.float32))
    xq, y = q8.rmsnorm_quantize(x, gamma, 1e-6, want_y=True)
    xq2, y2 = q8.rmsnorm_quantize(x, gamma, 1e-6, want_y=True)
    assert torch.equal(xq, xq2) and torch.equal(y, y2)
    W = dev(inputs.weights(out_dim, dim, seed=11))
    for n in (16, 3, 40):
        a = q8.matmul_q(W, xq[:n] if n <= n_tok else xq.repeat(3, 1)[:n], dim, out_dim)
        b = q8.matmul(W, y[:n] if n <= n_tok else y.repeat(3, 1)[:n], out_dim)
        assert torch.equal(a, b), n


def test_rmsnorm_quantize_argument_errors(q8):
    x = dev(inputs.normal((2, 64), seed=12))
    xq = torch.empty((2, 2 * QB), dtype=torch.uint8, device=DEV)
    for eps in (0.0, -1.0, float("nan"), float("inf")):
        assert q8.q8_rmsnorm_quantize(xq, None, x, None, 64, 2, eps) == q8.Q8_EINVAL
    assert q8.q8_rmsnorm_quantize(xq, None, x, None, 48, 2, 1e-6) == q8.Q8_EINVAL
    assert q8.q8_rmsnorm_quantize(None, None, x, None, 64, 2, 1e-6) == q8.Q8_EINVAL
    assert q8.q8_rmsnorm_quantize(xq, None, x.data_ptr() + 4, None, 64, 2, 1e-6) == q8.Q8_EALIGN
    assert q8.q8_rmsnorm_quantize(xq, None, x, None, 64, 0, 1e-6) == 0
    assert q8.q8_rmsnorm_quantize(xq, None, x, None, 64, 2, 1e-6) == 0
    assert q8.q8_last_error() == 0
