"""GPU parity of the routed expert FFN around the routed matmul (q8_moe_ffn) and
of its elementwise steps (q8_swiglu, q8_moe_combine), through the C ABI, against
the CPU oracle.

Tolerances, each derived from the arithmetic:

* SwiGLU: fp32 on the GPU (expf within 2 ulp, then three correctly rounded
  operations), double rounded once on the oracle side: at most 4 ulp, i.e.
  2^-21 |mid| (plus 1e-37 for results in the subnormal range).
* Weighted sum: k fp32 products and k fp32 sums, each within 2^-24 of a
  partial sum bounded by sum_j |w_j y_j|: 2k 2^-24 sum_j |w_j y_j|.
* FFN (oracle.ffn_tolerance): for every pair, the down projection's bound
  1e-4 B + 1e-6 (B the sum of |block terms|); 2^-10 B for a block whose binary16
  scale rounds the other way (one binary16 step); one quantisation step d for
  every mid value whose oracle quotient mid/d lies within 1e-3 of a rounding tie
  (the GPU's gate and up differ from the oracle's by fp32 rounding, far less
  than 1e-3 d, so codes can differ only there); then the weighted sum as above.
  An exactly constructed instance needs none of the allowances but the first.
"""
import numpy as np
import pytest

import inputs
import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
QK, QB = 32, 34
DEV = "cuda:0"
GUARD = 64


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


def blocks(d_bits, q):
    """Raw Q8_0 rows from binary16 scale bits [rows, nb] and quants [rows, nb, 32]."""
    rows, nb = d_bits.shape
    out = np.empty((rows, nb, QB), np.uint8)
    out[..., 0] = (d_bits & 0xFF).astype(np.uint8)
    out[..., 1] = (d_bits >> 8).astype(np.uint8)
    out[..., 2:] = q.astype(np.int8).view(np.uint8)
    return out.reshape(rows, nb * QB)


def gpu_ffn(q8, Wg, Wu, Wd, n_exp, gu_stride, d_stride, ids, w, x, mid_dim, out_dim, limit):
    n_tok = x.shape[0]
    k = ids.shape[1]
    buf = torch.full((n_tok * out_dim + GUARD,), float("nan"), dtype=torch.float32, device=DEV)
    rc = q8.q8_moe_ffn(buf, Wg, Wu, Wd, n_exp, gu_stride, d_stride, dev(ids), dev(w), k, x.shape[1], mid_dim,
                       out_dim, limit, dev(x), n_tok)
    assert rc == 0, f"{q8.q8_strerror(rc)} {q8.q8_last_cuda_error()}"
    h = buf.cpu().numpy()
    assert np.all(np.isnan(h[n_tok * out_dim:])), "guard band after the output was written"
    got = h[:n_tok * out_dim].reshape(n_tok, out_dim)
    assert not np.any(np.isnan(got)), "FFN output element not written"
    return got


def assert_ffn_close(got, r, tol, what):
    err = np.abs(got.astype(np.float64) - r["out"])
    bad = err > tol
    assert not np.any(bad), (f"{what}: {bad.sum()} outputs out of tolerance, worst err {err.max():.3e} "
                             f"at {np.unravel_index(np.argmax(err - tol), err.shape)}")


# ------------------------------------------------------------------ elementwise steps
@pytest.mark.parametrize("n", [4099, (1 << 20) + 2])
@pytest.mark.parametrize("limit", [10.0, 0.0])
def test_swiglu_parity(q8, o, n, limit):
    g = np.random.default_rng(n)
    gate = (8 * g.standard_normal(n)).astype(np.float32)
    up = (8 * g.standard_normal(n)).astype(np.float32)
    special = np.array([0.0, -0.0, 1000.0, -1000.0, 1e30, -1e30, 88.0, -88.0, 10.0, -10.0, 1e-30, -104.0],
                       np.float32)
    gate[:special.size] = special
    up[:special.size] = np.float32(3.0)
    gate[-3:], up[-3:] = np.float32(-20.0), np.float32(-50.0)   # the ragged tail too
    ref = o.swiglu(gate, up, limit).astype(np.float64)
    buf = torch.full((n + GUARD,), float("nan"), dtype=torch.float32, device=DEV)
    assert q8.q8_swiglu(buf, dev(gate), dev(up), n, limit) == 0
    h = buf.cpu().numpy()
    assert np.all(np.isnan(h[n:]))
    got = h[:n].astype(np.float64)
    err = np.abs(got - ref)
    assert np.all(err <= 2.0 ** -21 * np.abs(ref) + 1e-37), f"worst {err.max():.3e} at {np.argmax(err)}"


@pytest.mark.parametrize("dim", [4096, 33])
@pytest.mark.parametrize("k", [6, 1])
def test_combine_parity(q8, o, dim, k):
    n_tok = 37
    g = np.random.default_rng(dim + k)
    y = g.standard_normal((n_tok * k, dim)).astype(np.float32)
    w = g.random(n_tok * k).astype(np.float32)
    ref, bound = o.combine(y, w, n_tok, k)
    buf = torch.full((n_tok * dim + GUARD,), float("nan"), dtype=torch.float32, device=DEV)
    yd, wd = dev(y), dev(w)
    assert q8.q8_moe_combine(buf, yd, wd, n_tok, k, dim) == 0
    h = buf.cpu().numpy()
    assert np.all(np.isnan(h[n_tok * dim:]))
    got = h[:n_tok * dim].reshape(n_tok, dim).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2 * k * 2.0 ** -24 * bound + 1e-37)
    again = torch.empty((n_tok, dim), dtype=torch.float32, device=DEV)
    assert q8.q8_moe_combine(again, yd, wd, n_tok, k, dim) == 0
    assert np.array_equal(again.cpu().numpy(), got.astype(np.float32))


# ------------------------------------------------------------------ the routed FFN
def exact_instance(g, n_exp, in_dim, mid_dim, out_dim, n_tok, k):
    """An FFN whose every step is exact: x[t] = 127 e_{c_t}; every weight scale 1; block 0
    of each gate row all 1 (gate = 127, silu(127) = 127 in fp32); up = 127 q_up[o][0][c_t]
    with a +/-127 heading every 32-row block, so mid = 16129 q_up quantises to scale 16129
    (stored as 16128) and quants q_up; y = 16128 Q_down q_up exactly in integers."""
    nbi, nbm = in_dim // QK, mid_dim // QK
    one = np.uint16(0x3C00)
    qg = g.integers(-127, 128, size=(n_exp * mid_dim, nbi, QK))
    qg[:, 0, :] = 1
    qu = g.integers(-127, 128, size=(n_exp * mid_dim, nbi, QK))
    qu[::QK, 0, :] = 127 * g.choice([-1, 1], size=(n_exp * mid_dim // QK, QK))
    qd = g.integers(-127, 128, size=(n_exp * out_dim, nbm, QK))
    Wg = blocks(np.full((n_exp * mid_dim, nbi), one), qg)
    Wu = blocks(np.full((n_exp * mid_dim, nbi), one), qu)
    Wd = blocks(np.full((n_exp * out_dim, nbm), one), qd)
    ids = np.stack([g.choice(n_exp, size=k, replace=False) for _ in range(n_tok)]).astype(np.int32)
    w = g.choice([0.25, -0.5, 1.0, 2.0, 0.75], size=(n_tok, k)).astype(np.float32)
    c = g.integers(0, QK, size=n_tok)
    x = np.zeros((n_tok, in_dim), np.float32)
    x[np.arange(n_tok), c] = 127.0
    # exact y per pair and the bound of its block terms
    qu_t = qu.reshape(n_exp, mid_dim, nbi, QK)
    qd_t = qd.reshape(n_exp, out_dim, nbm, QK)
    y = np.empty((n_tok * k, out_dim), np.int64)
    yb = np.empty((n_tok * k, out_dim), np.float64)
    for t in range(n_tok):
        for j in range(k):
            e = int(ids[t, j])
            qmid = qu_t[e, :, 0, c[t]].reshape(nbm, QK)
            terms = 16128 * np.einsum("obi,bi->ob", qd_t[e], qmid)
            y[t * k + j], yb[t * k + j] = terms.sum(1), np.abs(terms).sum(1).astype(np.float64)
    return Wg.reshape(-1), Wu.reshape(-1), Wd.reshape(-1), ids, w, x, y, yb


@pytest.mark.parametrize("n_exp,in_dim,mid_dim,out_dim,n_tok,k", [
    (5, 64, 96, 48, 4, 2),          # in_dim/32 not a multiple of 8: the generic kernel
    (7, 256, 256, 200, 6, 3),       # routed GEMV
    (8, 256, 256, 136, 512, 2),     # 1024 pairs: the tensor-core class
])
def test_moe_ffn_exact_instance(q8, o, n_exp, in_dim, mid_dim, out_dim, n_tok, k):
    g = np.random.default_rng(n_exp * 1000 + n_tok)
    Wg, Wu, Wd, ids, w, x, y, yb = exact_instance(g, n_exp, in_dim, mid_dim, out_dim, n_tok, k)
    gu, ds = mid_dim * (in_dim // QK) * QB, out_dim * (mid_dim // QK) * QB
    got = gpu_ffn(q8, dev(Wg), dev(Wu), dev(Wd), n_exp, gu, ds, ids, w, x, mid_dim, out_dim, 0.0)
    assert q8.q8_last_error() == 0
    wt = w.astype(np.float64)
    exact = np.einsum("tj,tjo->to", wt, y.reshape(n_tok, k, out_dim).astype(np.float64))
    ybound = yb.reshape(n_tok, k, out_dim)
    tol = np.einsum("tj,tjo->to", np.abs(wt), 1e-4 * ybound + 1e-6) + \
        2 * k * 2.0 ** -24 * np.einsum("tj,tjo->to", np.abs(wt), ybound)
    assert np.all(np.abs(got - exact) <= tol)
    if n_tok <= 8:   # and the oracle agrees (its own pins cover the larger case)
        r = o.moe_ffn(Wg, Wu, Wd, n_exp, gu, ds, ids, w, in_dim, mid_dim, out_dim, 0.0, x)
        assert np.all(np.abs(got - r["out"]) <= 2 * tol)


@pytest.mark.parametrize("n_exp,in_dim,mid_dim,out_dim,n_tok,k,limit", [
    (16, 512, 256, 384, 24, 4, 10.0),    # routed GEMV, clamp on
    (16, 512, 256, 384, 24, 4, 0.0),     # clamp off
    (64, 1024, 512, 256, 40, 6, 10.0),   # one routing: pair items of 224, 224, 64 rows write mid as Q8_0
    (64, 1024, 480, 256, 40, 6, 10.0),   # mid_dim % 256 != 0: pair items (224, 224, 32 rows) write fp32 mid
    (8, 256, 256, 256, 512, 2, 10.0),    # tensor-core class for gate, up and down
    (6, 96, 64, 40, 5, 2, 10.0),         # generic kernel
])
def test_moe_ffn_random(q8, o, n_exp, in_dim, mid_dim, out_dim, n_tok, k, limit):
    seed = n_exp + in_dim + n_tok
    Wg = inputs.weights(n_exp * mid_dim, in_dim, seed=seed).reshape(-1)
    Wu = inputs.weights(n_exp * mid_dim, in_dim, seed=seed + 1).reshape(-1)
    Wd = inputs.weights(n_exp * out_dim, mid_dim, seed=seed + 2).reshape(-1)
    gu, ds = mid_dim * (in_dim // QK) * QB, out_dim * (mid_dim // QK) * QB
    ids = inputs.route_uniform(n_tok, k, n_exp, seed=seed)
    g = np.random.default_rng(seed)
    w = g.random((n_tok, k)).astype(np.float32)
    x = inputs.normal((n_tok, in_dim), seed=seed, p_out=0.01)
    got = gpu_ffn(q8, dev(Wg), dev(Wu), dev(Wd), n_exp, gu, ds, ids, w, x, mid_dim, out_dim, limit)
    assert q8.q8_last_error() == 0
    r = o.moe_ffn(Wg, Wu, Wd, n_exp, gu, ds, ids, w, in_dim, mid_dim, out_dim, limit, x)
    assert r["flag"] == 0
    if limit > 0:   # the clamp is exercised: without it the oracle's mid differs
        r0 = o.moe_ffn(Wg, Wu, Wd, n_exp, gu, ds, ids, w, in_dim, mid_dim, out_dim, 0.0, x)
        assert not np.array_equal(r0["mid"], r["mid"])
    assert_ffn_close(got, r, oracle.ffn_tolerance(r, Wd, ds, ids, w, mid_dim, out_dim), "moe ffn")


def test_moe_ffn_decode_config_sampled(q8, o):
    """The routed decode layer at full size: 256 experts, gate/up [2048 x 4096], down
    [4096 x 2048], 64 tokens, uniform top-6, clamp 10; the oracle on sampled tokens
    (tokens are independent), every output finite."""
    n_exp, n_tok, k, in_dim, mid_dim, out_dim = 256, 64, 6, 4096, 2048, 4096
    ids = inputs.route_uniform(n_tok, k, n_exp, seed=0)
    Wg = inputs.weights(n_exp * mid_dim, in_dim, seed=0).reshape(-1)
    Wu = inputs.weights(n_exp * mid_dim, in_dim, seed=10).reshape(-1)
    Wd = inputs.weights(n_exp * out_dim, mid_dim, seed=1).reshape(-1)
    gu, ds = mid_dim * (in_dim // QK) * QB, out_dim * (mid_dim // QK) * QB
    w = np.random.default_rng(0).random((n_tok, k)).astype(np.float32)
    x = inputs.normal((n_tok, in_dim), seed=0)
    got = gpu_ffn(q8, dev(Wg), dev(Wu), dev(Wd), n_exp, gu, ds, ids, w, x, mid_dim, out_dim, 10.0)
    assert q8.q8_last_error() == 0
    for t in (0, 31, 63):
        sl = slice(t, t + 1)
        r = o.moe_ffn(Wg, Wu, Wd, n_exp, gu, ds, ids[sl], w[sl], in_dim, mid_dim, out_dim, 10.0, x[sl])
        assert_ffn_close(got[sl], r, oracle.ffn_tolerance(r, Wd, ds, ids[sl], w[sl], mid_dim, out_dim), f"token {t}")


@pytest.mark.parametrize("mid_dim", [128, 256])   # down on the generic kernel / the one-routing path
def test_moe_ffn_bad_id_and_determinism(q8, o, mid_dim):
    n_exp, in_dim, out_dim, n_tok, k = 6, 256, 96, 5, 3
    Wg = inputs.weights(n_exp * mid_dim, in_dim, seed=31).reshape(-1)
    Wu = inputs.weights(n_exp * mid_dim, in_dim, seed=32).reshape(-1)
    Wd = inputs.weights(n_exp * out_dim, mid_dim, seed=33).reshape(-1)
    gu, ds = mid_dim * (in_dim // QK) * QB, out_dim * (mid_dim // QK) * QB
    ids = inputs.route_uniform(n_tok, k, n_exp, seed=34)
    ids[1, 2], ids[3, 0] = 6, -1
    w = np.random.default_rng(35).random((n_tok, k)).astype(np.float32)
    x = inputs.normal((n_tok, in_dim), seed=36)
    a = gpu_ffn(q8, dev(Wg), dev(Wu), dev(Wd), n_exp, gu, ds, ids, w, x, mid_dim, out_dim, 10.0)
    assert q8.q8_last_error() == q8.Q8_ERANGE
    r = o.moe_ffn(Wg, Wu, Wd, n_exp, gu, ds, ids, w, in_dim, mid_dim, out_dim, 10.0, x)
    assert r["flag"] == 1
    assert_ffn_close(a, r, oracle.ffn_tolerance(r, Wd, ds, np.where(ids < 0, 0, ids % n_exp), w, mid_dim, out_dim),
                     "bad id")
    b = gpu_ffn(q8, dev(Wg), dev(Wu), dev(Wd), n_exp, gu, ds, ids, w, x, mid_dim, out_dim, 10.0)
    assert q8.q8_last_error() == q8.Q8_ERANGE
    assert np.array_equal(a, b)


def test_moe_ffn_argument_errors(q8):
    n_exp, in_dim, mid_dim, out_dim, n_tok, k = 4, 64, 32, 16, 2, 2
    Wg = dev(inputs.weights(n_exp * mid_dim, in_dim, seed=41))
    Wd = dev(inputs.weights(n_exp * out_dim, mid_dim, seed=42))
    gu, ds = mid_dim * 2 * QB, out_dim * QB
    ids = dev(np.array([[0, 1], [2, 3]], np.int32))
    w = dev(np.ones((2, 2), np.float32))
    x = dev(inputs.normal((n_tok, in_dim), seed=43))
    out = torch.empty((n_tok, out_dim), dtype=torch.float32, device=DEV)
    call = lambda **kw: q8.q8_moe_ffn(*[kw.get(n, v) for n, v in (
        ("out", out), ("Wg", Wg), ("Wu", Wg), ("Wd", Wd), ("n_exp", n_exp), ("gu", gu), ("ds", ds), ("ids", ids),
        ("w", w), ("k", k), ("in_dim", in_dim), ("mid_dim", mid_dim), ("out_dim", out_dim), ("limit", 10.0),
        ("x", x), ("n_tok", n_tok))])
    assert call() == 0
    assert q8.q8_last_error() == 0
    assert call(limit=float("nan")) == q8.Q8_EINVAL
    assert call(limit=-1.0) == q8.Q8_EINVAL
    assert call(mid_dim=48) == q8.Q8_EINVAL            # not a multiple of 32
    assert call(k=5) == q8.Q8_EINVAL                   # more slots than experts
    assert call(gu=gu - 16) == q8.Q8_EINVAL            # stride shorter than a matrix
    assert call(ds=ds + 8) == q8.Q8_EALIGN             # stride not a multiple of 16
    assert call(w=None) == q8.Q8_EINVAL
    assert call(x=x.data_ptr() + 4) == q8.Q8_EALIGN
    assert call(n_tok=0) == 0
    m = torch.empty(8, device=DEV)
    assert q8.q8_swiglu(m, m, m, 8, float("nan")) == q8.Q8_EINVAL
    assert q8.q8_swiglu(m, m, m, 0, 1.0) == 0
    assert q8.q8_moe_combine(m, m, m, 1, 0, 8) == q8.Q8_EINVAL
