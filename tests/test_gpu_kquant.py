"""GPU parity of the second weight format: Q2_K / Q4_K rows against Q8_K activations,
through the C ABI, against the CPU oracle.

The Q8_K quantiser must be bit-exact (fp32 d, int8 quants, and the int16 sums of each
16 quants stored with them).  Products must satisfy
|gpu - oracle| <= 1e-4 * sum over sub-blocks |d_x| (|d sc isum| + |dmin m xsum|) + 1e-6
element by element.  Outputs are poisoned with NaN and followed by a guard band.
"""
import numpy as np
import pytest

import inputs
import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
QKK = 256
GUARD = 64
FMTS = (2, 4)   # Q2_K, Q4_K


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


DEV = "cuda:0"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def poisoned(n):
    return torch.full((n + GUARD,), float("nan"), dtype=torch.float32, device=DEV)


def fetch(buf, n, shape):
    h = buf.cpu().numpy()
    assert np.all(np.isnan(h[n:])), "guard band after the output was written"
    return h[:n].reshape(shape)


def assert_close(got, ref, bound, what=""):
    assert not np.any(np.isnan(got)), f"{what}: output element not written (NaN poison survived)"
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    tol = oracle.tolerance(bound)
    bad = err > tol
    assert not np.any(bad), (f"{what}: {bad.sum()} outputs out of tolerance, worst err {err.max():.3e} "
                             f"at {np.unravel_index(np.argmax(err - tol), err.shape)}")


def _acts(g, n_tok, in_dim):
    """N(0,1) rows with zero blocks, exact ties and wide magnitudes mixed in."""
    x = g.standard_normal((n_tok, in_dim)).astype(np.float32)
    xb = x.reshape(n_tok, -1, QKK)
    kinds = g.integers(0, 5, size=xb.shape[:2])
    for t, b in zip(*np.nonzero(kinds == 0)):
        xb[t, b] = 0.0
    for t, b in zip(*np.nonzero(kinds == 1)):
        d = np.float32(2.0 ** g.integers(-12, 4))
        v = (g.integers(0, 126, QKK) + 0.5) * np.where(g.random(QKK) < .5, -1, 1)
        v[0] = 127
        xb[t, b] = (d * v).astype(np.float32)
    for t, b in zip(*np.nonzero(kinds == 2)):
        xb[t, b] *= np.float32(np.exp(g.uniform(-20, 20)))
    return x


# ------------------------------------------------------------------ quantiser
@pytest.mark.parametrize("n_tok,in_dim", [(1, 256), (3, 768), (16, 4096), (37, 2048)])
def test_q8k_quantiser_bitexact(q8, o, n_tok, in_dim):
    x = _acts(np.random.default_rng(n_tok * 7 + in_dim), n_tok, in_dim)
    d_ref, q_ref = o.quantize_q8k(x)
    blk = q8.quantize_q8k(dev(x)).cpu().numpy().reshape(n_tok, in_dim // QKK, 292)
    d = blk[..., :4].copy().view(np.float32)[..., 0]
    q = blk[..., 4:260].copy().view(np.int8).reshape(n_tok, in_dim)
    sums = blk[..., 260:].copy().view(np.int16)
    assert np.array_equal(d.view(np.uint32), d_ref.view(np.uint32))
    assert np.array_equal(q, q_ref)
    assert np.array_equal(sums.astype(np.int64), q_ref.reshape(n_tok, -1, 16, 16).astype(np.int64).sum(-1))


# ------------------------------------------------------------------ dense product
KQ_SHAPES = [
    (256, 1, 1), (256, 7, 2), (512, 33, 3), (1024, 100, 8), (2048, 64, 9), (768, 300, 16),
    (4096, 40, 17),   # two token groups, ragged
    (1280, 130, 40),  # three token groups
]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("in_dim,out_dim,n_tok", KQ_SHAPES)
def test_kq_matmul_parity(q8, o, fmt, in_dim, out_dim, n_tok):
    W = inputs.kq_weights(out_dim, in_dim, fmt, seed=in_dim + out_dim)
    x = _acts(np.random.default_rng(n_tok + 5 * out_dim), n_tok, in_dim)
    ref, bound = o.kq_matmul(W, fmt, x, out_dim)
    buf = poisoned(n_tok * out_dim)
    rc = q8.q8_kq_matmul(buf, dev(W), fmt, in_dim, out_dim, dev(x), n_tok)
    assert rc == 0, q8.q8_strerror(rc)
    assert q8.q8_last_error() == 0
    assert_close(fetch(buf, n_tok * out_dim, (n_tok, out_dim)), ref, bound, f"kq{fmt} {in_dim}x{out_dim}x{n_tok}")


def test_kq_matmul_direct_kernel_cases(q8, o):
    """Rows the staged kernel does not take: Q2_K rows that are not 16-byte multiples (in_dim 1280), a
    Q2_K matrix only 4-byte aligned, and Q4_K rows longer than a shared-memory slot (in_dim 73728)."""
    cases = [(2, 1280, 50, 5, 0), (2, 1024, 40, 3, 4), (4, 73728, 6, 3, 0)]
    for fmt, in_dim, out_dim, n_tok, offset in cases:
        W = inputs.kq_weights(out_dim, in_dim, fmt, seed=in_dim + offset)
        x = _acts(np.random.default_rng(in_dim), n_tok, in_dim)
        ref, bound = o.kq_matmul(W, fmt, x, out_dim)
        Wd = torch.zeros(W.nbytes + 16, dtype=torch.uint8, device=DEV)
        Wd[offset:offset + W.nbytes] = dev(W.reshape(-1))
        buf = poisoned(n_tok * out_dim)
        rc = q8.q8_kq_matmul(buf, Wd.data_ptr() + offset, fmt, in_dim, out_dim, dev(x), n_tok)
        assert rc == 0, q8.q8_strerror(rc)
        assert q8.q8_last_error() == 0
        assert_close(fetch(buf, n_tok * out_dim, (n_tok, out_dim)), ref, bound, f"kq{fmt} direct {in_dim}+{offset}")


@pytest.mark.parametrize("fmt", FMTS)
def test_kq_matmul_decode_projection_full(q8, o, fmt):
    """A routed expert's gate projection, 4096 -> 2048, one token: every output."""
    W = inputs.kq_weights(2048, 4096, fmt, seed=11)
    x = inputs.normal((1, 4096), seed=12, p_out=0.01)
    ref, bound = o.kq_matmul(W, fmt, x, 2048)
    assert_close(q8.kq_matmul(dev(W), fmt, dev(x), 2048).cpu().numpy(), ref, bound, f"kq{fmt} decode")


@pytest.mark.parametrize("fmt", FMTS)
def test_kq_matmul_repeatable(q8, fmt):
    W = dev(inputs.kq_weights(300, 1024, fmt, seed=3))
    x = dev(inputs.normal((20, 1024), seed=4))
    a = q8.kq_matmul(W, fmt, x, 300)
    b = q8.kq_matmul(W, fmt, x, 300)
    assert torch.equal(a, b)


# ------------------------------------------------------------------ routed experts
def _gpu_kq_moe(q8, Wd, fmt, n_exp, stride, ids, x, x_per_pair, out_dim):
    n_tok, k = ids.shape
    n = n_tok * k * out_dim
    buf = poisoned(n)
    rc = q8.q8_kq_moe_matmul(buf, Wd, fmt, n_exp, stride, dev(ids), k, x.shape[1], out_dim, dev(x),
                             int(x_per_pair), n_tok)
    assert rc == 0, q8.q8_strerror(rc)
    return fetch(buf, n, (n_tok * k, out_dim))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("x_per_pair", [0, 1])
def test_kq_moe_every_output(q8, o, fmt, x_per_pair):
    """37 tokens, top-3 of 16 experts: groups of 1-16+ rows (both GEMV classes), every output."""
    n_exp, in_dim, out_dim, n_tok, k = 16, 512, 72, 37, 3
    stride = out_dim * q8.q8_kq_row_bytes(in_dim, fmt)
    Wall = inputs.kq_weights(n_exp * out_dim, in_dim, fmt, seed=21).reshape(-1)
    ids = inputs.route_zipf(n_tok, k, n_exp, seed=22)
    x = _acts(np.random.default_rng(23), n_tok * k if x_per_pair else n_tok, in_dim)
    ref, bound, flag = o.kq_moe(Wall, fmt, n_exp, stride, ids, in_dim, out_dim, x, x_per_pair)
    assert flag == 0
    counts = np.bincount(ids.reshape(-1), minlength=n_exp)
    assert counts.max() > 8 and counts[counts > 0].min() <= 8       # both GEMV classes run
    got = _gpu_kq_moe(q8, dev(Wall), fmt, n_exp, stride, ids, x, x_per_pair, out_dim)
    assert q8.q8_last_error() == 0
    assert_close(got, ref, bound, f"kq{fmt} moe per_pair={x_per_pair}")


@pytest.mark.parametrize("fmt", FMTS)
def test_kq_moe_bad_id(q8, o, fmt):
    n_exp, in_dim, out_dim, n_tok, k = 4, 256, 24, 3, 2
    stride = out_dim * q8.q8_kq_row_bytes(in_dim, fmt) + 16
    Wall = np.zeros(n_exp * stride, np.uint8)
    rows = inputs.kq_weights(n_exp * out_dim, in_dim, fmt, seed=31).reshape(n_exp, -1)
    for e in range(n_exp):
        Wall[e * stride:e * stride + rows.shape[1]] = rows[e]
    ids = np.array([[0, 7], [-1, 2], [3, 1]], dtype=np.int32)
    x = _acts(np.random.default_rng(32), n_tok, in_dim)
    ref, bound, flag = o.kq_moe(Wall, fmt, n_exp, stride, ids, in_dim, out_dim, x, 0)
    assert flag == 1
    got = _gpu_kq_moe(q8, dev(Wall), fmt, n_exp, stride, ids, x, 0, out_dim)
    assert q8.q8_last_error() == q8.Q8_ERANGE
    assert np.all(got[[1, 2]] == 0)
    assert_close(got, ref, bound, f"kq{fmt} moe bad id")


@pytest.mark.parametrize("fmt", FMTS)
def test_kq_moe_decode_config_sampled(q8, o, fmt):
    """The routed experts' decode shape: 256 experts of [2048 x 4096], 64 tokens, uniform top-6;
    the outputs of 8 pairs checked in full against the oracle's dense product of their expert."""
    n_exp, in_dim, out_dim, n_tok, k = 256, 4096, 2048, 64, 6
    stride = out_dim * q8.q8_kq_row_bytes(in_dim, fmt)
    Wd = torch.empty(n_exp * stride, dtype=torch.uint8, device=DEV)
    chunk = 32
    for e0 in range(0, n_exp, chunk):
        Wd[e0 * stride:(e0 + chunk) * stride] = dev(
            inputs.kq_weights(chunk * out_dim, in_dim, fmt, seed=41 + e0).reshape(-1))
    ids = inputs.route_uniform(n_tok, k, n_exp, seed=42)
    x = inputs.normal((n_tok, in_dim), seed=43, p_out=0.01)
    got = _gpu_kq_moe(q8, Wd, fmt, n_exp, stride, ids, x, 0, out_dim)
    assert q8.q8_last_error() == 0
    for p in np.random.default_rng(44).choice(n_tok * k, size=8, replace=False):
        e = int(ids.reshape(-1)[p])
        We = Wd[e * stride:(e + 1) * stride].cpu().numpy()
        ref, bound = o.kq_matmul(We, fmt, x[p // k][None], out_dim)
        assert_close(got[p][None], ref, bound, f"kq{fmt} pair {p} expert {e}")


@pytest.mark.parametrize("fmt", FMTS)
def test_kq_moe_down_shape_sampled(q8, o, fmt):
    """The routed down projection's shape: 256 experts of [4096 x 2048] on per-pair rows, 64
    tokens, uniform top-6.  Short rows fill items of 28 (Q4_K) or 56 (Q2_K) rows, the last of
    each expert ragged (4096 = 146 x 28 + 8); 8 pairs checked in full against the oracle."""
    n_exp, in_dim, out_dim, n_tok, k = 256, 2048, 4096, 64, 6
    stride = out_dim * q8.q8_kq_row_bytes(in_dim, fmt)
    Wd = torch.empty(n_exp * stride, dtype=torch.uint8, device=DEV)
    chunk = 32
    for e0 in range(0, n_exp, chunk):
        Wd[e0 * stride:(e0 + chunk) * stride] = dev(
            inputs.kq_weights(chunk * out_dim, in_dim, fmt, seed=51 + e0).reshape(-1))
    ids = inputs.route_uniform(n_tok, k, n_exp, seed=52)
    x = inputs.normal((n_tok * k, in_dim), seed=53, p_out=0.01)
    got = _gpu_kq_moe(q8, Wd, fmt, n_exp, stride, ids, x, 1, out_dim)
    assert q8.q8_last_error() == 0
    for p in np.random.default_rng(54).choice(n_tok * k, size=8, replace=False):
        e = int(ids.reshape(-1)[p])
        We = Wd[e * stride:(e + 1) * stride].cpu().numpy()
        ref, bound = o.kq_matmul(We, fmt, x[p][None], out_dim)
        assert_close(got[p][None], ref, bound, f"kq{fmt} down pair {p} expert {e}")
