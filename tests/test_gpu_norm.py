"""GPU parity of RMSNorm feeding the quantiser (q8_rmsnorm_quantize) through the C
ABI, against the CPU oracle.

* The quantised rows must be bit for bit the activation quantiser (q8_quantize_act,
  itself bit-exact to the oracle) applied to the kernel's own normalised rows y:
  the fused quantiser is the a1 quantiser.
* y against the oracle's y (double, rounded once): the kernel's sum of squares has
  relative error at most n_s 2^-24 with n_s = 8 ceil(dim/2048) + 14 (its fixed
  reduction order); the mean, + eps, sqrt, reciprocal, two products and the
  oracle's own rounding add at most 7 more roundings, and sqrt halves the sum's
  error: ((n_s + 2) / 2 + 5) 2^-24 to first order; rho adds one more 2^-24 for the
  second-order terms (plus 1e-37 near the subnormal range).  This holds while the
  squares neither overflow nor underflow in fp32.
* The oracle's quantised rows then differ only where that error can move a
  decision: a quant by 1 where the oracle's |y/d| lies within a window of a
  rounding tie, the binary16 scale by one step where the oracle's fp32 d lies
  within 4 rho of a binary16 rounding midpoint.  The window is
  max(1e-3, 3 (2 rho + 2^-22) 127), three times the largest movement of y/d.
"""
import math

import numpy as np
import pytest

import inputs
import oracle

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


def rho(dim):
    n_s = 8 * math.ceil(dim / 2048) + 14
    return ((n_s + 2) / 2 + 6) * 2.0 ** -24


def split(xq, nb):
    r = xq.reshape(xq.shape[0], nb, QB)
    d = r[..., 0].astype(np.uint16) | (r[..., 1].astype(np.uint16) << 8)
    q = r[..., 2:].copy().view(np.int8).astype(np.int32)
    return d, q


def f16_near_midpoint(d32, rel):
    """True where the fp32 value lies within rel (relative) of a binary16 rounding midpoint."""
    d = d32.astype(np.float64)
    h = d32.astype(np.float16).astype(np.float64)
    up = np.nextafter(d32.astype(np.float16), np.float16(np.inf)).astype(np.float64)
    dn = np.nextafter(d32.astype(np.float16), np.float16(0)).astype(np.float64)
    mids = np.stack([(h + up) / 2, (h + dn) / 2])
    return np.any(np.abs(mids - d) <= rel * np.abs(d), axis=0)


def check(q8, o, x, gamma, eps):
    n_tok, dim = x.shape
    nb = dim // QK
    xq, y = q8.rmsnorm_quantize(dev(x), None if gamma is None else dev(gamma), eps, want_y=True)
    assert q8.q8_last_error() == 0
    # the fused quantiser is the activation quantiser of the kernel's own y
    assert torch.equal(xq, q8.quantize_act(y))
    xq_o, y_o = o.rmsnorm_quantize(x, gamma, eps)
    yg = y.cpu().numpy().astype(np.float64)
    r = rho(dim)
    err = np.abs(yg - y_o)
    assert np.all(err <= r * np.abs(y_o) + 1e-37), f"y: worst relative {np.max(err / (np.abs(y_o) + 1e-30)):.3e}"
    dg, qg = split(xq.cpu().numpy(), nb)
    do, qo = split(xq_o, nb)
    d32 = np.abs(y_o.reshape(n_tok, nb, QK)).max(-1).astype(np.float32) / np.float32(127.0)
    near_mid = f16_near_midpoint(d32, 4 * r)
    dgf = dg.view(np.float16).astype(np.float64)
    dof = do.view(np.float16).astype(np.float64)
    step = np.abs(np.nextafter(do.view(np.float16), np.float16(np.inf)).astype(np.float64) - dof)
    assert np.all((dg == do) | (near_mid & (np.abs(dgf - dof) <= step))), "binary16 scale differs away from a midpoint"
    window = max(1e-3, 3 * (2 * r + 2.0 ** -22) * 127)
    with np.errstate(divide="ignore", invalid="ignore"):
        quo = np.abs(y_o.reshape(n_tok, nb, QK) / d32[..., None].astype(np.float64))
    near_tie = np.abs(quo - np.floor(quo) - 0.5) < window
    diff = qg != qo
    assert np.all(np.abs(qg - qo) <= 1)
    assert np.all(~diff | near_tie), f"{np.sum(diff & ~near_tie)} quants differ away from a tie"
    return xq, y


@pytest.mark.parametrize("dim,n_tok", [(4096, 37), (1024, 5), (96, 3), (32, 7), (2080, 4), (6144, 9), (16384, 2)])
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
