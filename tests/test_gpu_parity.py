"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Quantised activations must be bit-exact; matmul outputs must satisfy
|gpu - oracle| <= 1e-4 * sum_b |d_w d_x isum_b| + 1e-6 element by element.
Outputs are poisoned with NaN before every call and followed by a NaN guard
band that must stay untouched, so a kernel that skips rows or writes out of
bounds fails.
"""
import numpy as np
import pytest

import inputs
import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
QK, QB = 32, 34
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


def gpu_matmul(q8, W, x, out_dim):
    n_tok, in_dim = x.shape
    buf = poisoned(n_tok * out_dim)
    rc = q8.q8_matmul(buf, W, in_dim, out_dim, x, n_tok)
    assert rc == 0, f"{q8.q8_strerror(rc)} {q8.q8_last_cuda_error()}"
    assert q8.q8_last_error() == 0
    return fetch(buf, n_tok * out_dim, (n_tok, out_dim))


# ------------------------------------------------------------------ quantiser
def _special_x(g, n_tok, in_dim):
    x = g.standard_normal((n_tok, in_dim)).astype(np.float32)
    xb = x.reshape(n_tok, -1, QK)
    nb = xb.shape[1]
    kinds = g.integers(0, 6, size=(n_tok, nb))
    for t in range(n_tok):
        for b in range(nb):
            k = kinds[t, b]
            if k == 0:
                xb[t, b] = 0.0                                              # all-zero block
            elif k == 1:
                d = np.float32(2.0 ** g.integers(-20, 4))                   # exact ties (m + 1/2) * d
                v = (g.integers(0, 126, QK) + 0.5) * np.where(g.random(QK) < .5, -1, 1)
                v[0] = 127
                xb[t, b] = (d * v).astype(np.float32)
            elif k == 2:
                xb[t, b] *= np.float32(1e-6)                                # subnormal binary16 scale
            elif k == 3:
                xb[t, b] *= np.float32(1e-40)                               # scale underflows
            elif k == 4:
                xb[t, b] *= np.float32(np.exp(g.uniform(-30, 30)))          # wide magnitudes
    return x


@pytest.mark.parametrize("n_tok,in_dim", [(1, 32), (3, 96), (16, 1024), (37, 4096), (5, 32768)])
def test_quantize_bit_exact(q8, o, n_tok, in_dim):
    g = np.random.default_rng(n_tok * 7 + in_dim)
    for x in (inputs.normal((n_tok, in_dim), seed=n_tok, p_out=0.01), _special_x(g, n_tok, in_dim)):
        ref = o.quantize(x)
        xq = torch.full((n_tok * (in_dim // QK) * QB + GUARD,), 0xAB, dtype=torch.uint8, device=DEV)
        assert q8.q8_quantize_act(xq, dev(x), in_dim, n_tok) == 0
        h = xq.cpu().numpy()
        assert np.all(h[-GUARD:] == 0xAB)
        got = h[:-GUARD].reshape(ref.shape)
        mism = np.argwhere(got != ref)
        assert mism.size == 0, f"{len(mism)} bytes differ, first at {mism[:3].tolist()}"


def test_quantize_prefill_size_bit_exact(q8, o):
    x = inputs.normal((512, 32768), seed=0)
    assert np.array_equal(q8.quantize_act(dev(x)).cpu().numpy(), o.quantize(x))


# ------------------------------------------------------------------ dense matmul, small and ragged
SHAPES = [
    (256, 16, 1), (512, 100, 3), (1024, 33, 16), (2048, 250, 17), (256, 1000, 64), (768, 77, 65),
    (4096, 40, 130), (8192, 24, 5), (1280, 131, 200),
    # prefill with nb % 8 != 0: weights expanded to an fp16 plane instead of read raw
    (2112, 130, 150),
    # one output tile with a long K: split over 32 CTAs, partial sums added in order
    (16384, 96, 20),
    # in_dim % 256 != 0: rows not 16-byte aligned (slow path)
    (32, 5, 1), (96, 19, 7), (160, 50, 20), (4000, 8, 2),
    # single and seven output rows (fewer rows than any tile or TMA box): the GEMV in
    # each mode, the tcgen05 GEMM on raw and on expanded weights
    (256, 1, 1), (1024, 7, 4), (4096, 1, 16), (512, 7, 100), (256, 1, 33), (2048, 1, 2100), (1024, 7, 20),
    # raw weights up to 2048 tokens (several token tiles, ragged last tile)
    (1024, 130, 1000), (2048, 1, 700),
    # in_dim 64 (two blocks a row): the slow path, and the tcgen05 GEMM with one K stage
    (64, 7, 1), (64, 1, 16), (64, 1, 20), (64, 130, 40), (64, 7, 300),
]


@pytest.mark.parametrize("in_dim,out_dim,n_tok", SHAPES)
def test_matmul_parity(q8, o, in_dim, out_dim, n_tok):
    Wh = inputs.weights(out_dim, in_dim, seed=in_dim + out_dim)
    xh = inputs.normal((n_tok, in_dim), seed=n_tok, p_out=0.01)
    ref, bound = o.matmul(Wh, xh, out_dim)
    got = gpu_matmul(q8, dev(Wh), dev(xh), out_dim)
    assert_close(got, ref, bound, f"matmul {in_dim}x{out_dim}x{n_tok}")


@pytest.mark.parametrize("n_tok,in_dim,out_dim", [(3, 4352, 300), (7, 4352, 130), (9, 4352, 150),
                                                   (13, 2816, 77), (16, 6400, 50)])
def test_planes_staging_ragged_chunks(q8, o, n_tok, in_dim, out_dim):
    """The GEMV's MMA modes staging pre-quantised activations from the planes (dense calls
    copy the token rows to shared memory in 16-byte pieces and build the fragments there):
    token counts that leave rows of an 8-token tile empty, and K chunks of 80 (one tile) or
    40 (two tiles) blocks with a ragged last chunk (136, 88 and 200 blocks)."""
    Wh = inputs.weights(out_dim, in_dim, seed=in_dim + n_tok)
    xh = inputs.normal((n_tok, in_dim), seed=n_tok + 5, p_out=0.01)
    ref, bound = o.matmul(Wh, xh, out_dim)
    xq = q8.quantize_act(dev(xh))
    got = q8.matmul_q(dev(Wh), xq, in_dim, out_dim).cpu().numpy()
    assert q8.q8_last_error() == 0
    assert_close(got, ref, bound, f"matmul_q {in_dim}x{out_dim}x{n_tok}")


@pytest.mark.parametrize("out_dim,n_tok", [(40000, 1), (40000, 16), (70000, 4), (70000, 16)])
def test_gemv_wide_outputs(q8, o, out_dim, n_tok):
    """Outputs wider than 152 x 14 sixteen-row sub-items: each CTA item holds 17 (out
    40000) or 29 (out 70000) sub-items, so the GEMV variants whose consumer warps hold two
    or three sub-items run.  Every output against the oracle."""
    in_dim = 256
    Wh = inputs.weights(out_dim, in_dim, seed=out_dim + n_tok)
    xh = inputs.normal((n_tok, in_dim), seed=n_tok, p_out=0.01)
    ref, bound = o.matmul(Wh, xh, out_dim)
    assert_close(gpu_matmul(q8, dev(Wh), dev(xh), out_dim), ref, bound, f"wide {out_dim} x {n_tok}")


@pytest.mark.parametrize("in_dim,out_dim,n_tok", [(1024, 300, 40), (1024, 200, 700), (2048, 70, 12)])
def test_matmul_q_matches_matmul_bitwise(q8, o, in_dim, out_dim, n_tok):
    """Pre-quantised activations give the same bits as fp32 ones: prefill with raw weights
    (40 tokens), with the fp16 weight plane (700 tokens), and the 9-16-token GEMV."""
    W = dev(inputs.weights(out_dim, in_dim, seed=5))
    x = dev(inputs.normal((n_tok, in_dim), seed=6))
    a = q8.matmul(W, x, out_dim)
    b = q8.matmul_q(W, q8.quantize_act(x), in_dim, out_dim)
    assert torch.equal(a, b)


@pytest.mark.parametrize("n_tok,in_dim,out_dim", [(1, 256, 100), (2, 1024, 333), (3, 512, 64), (8, 1024, 1000),
                                                   (8, 4096, 150), (5, 2048, 4100), (1, 16384, 40), (2, 8192, 77),
                                                   (16, 1024, 300), (12, 2048, 77), (9, 512, 5000)])
def test_fused_quantiser_matches_planes_bitwise(q8, n_tok, in_dim, out_dim):
    """Small dense calls quantise inside the GEMV; q8_matmul_q feeds the same GEMV
    from quantiser-kernel output.  Any difference in a quant or a scale (ties,
    subnormal and underflowing scales included) changes the result bits."""
    g = np.random.default_rng(in_dim + n_tok)
    W = dev(inputs.weights(out_dim, in_dim, seed=11))
    # special blocks reach binary16 overflow (inf scales, inf/nan outputs): compare bit patterns
    for xh in (inputs.normal((n_tok, in_dim), seed=n_tok, p_out=0.01), _special_x(g, n_tok, in_dim)):
        x = dev(xh)
        a = q8.matmul(W, x, out_dim)
        b = q8.matmul_q(W, q8.quantize_act(x), in_dim, out_dim)
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_integer_case_exact(q8):
    """All scales 1.0 and activations that quantise to themselves: exact integer product."""
    g = np.random.default_rng(3)
    in_dim, out_dim, n_tok = 512, 64, 20
    nb = in_dim // QK
    qw = g.integers(-127, 128, size=(out_dim, nb, QK))
    Wh = np.empty((out_dim, nb, QB), np.uint8)
    Wh[..., 0], Wh[..., 1] = 0x00, 0x3C
    Wh[..., 2:] = qw.astype(np.int8).view(np.uint8)
    qx = g.integers(-127, 128, size=(n_tok, nb, QK))
    qx[:, :, 0] = 127                                   # every block's max is 127: d = 1 exactly
    xh = qx.reshape(n_tok, in_dim).astype(np.float32)
    got = gpu_matmul(q8, dev(Wh.reshape(out_dim, -1)), dev(xh), out_dim)
    ref = xh.astype(np.int64) @ qw.reshape(out_dim, in_dim).T
    assert np.array_equal(got.astype(np.int64), ref)


def test_deterministic(q8):
    in_dim, out_dim, n_tok = 2048, 512, 100
    W = dev(inputs.weights(out_dim, in_dim, seed=8))
    x = dev(inputs.normal((n_tok, in_dim), seed=9))
    a = q8.matmul(W, x, out_dim)
    for _ in range(3):
        assert torch.equal(a, q8.matmul(W, x, out_dim))


# ------------------------------------------------------------------ the five workloads
def test_config1_single_matvec(q8, o):
    Wh = inputs.weights(1024, 4096, seed=0)
    xh = inputs.normal((1, 4096), seed=0)
    ref, bound = o.matmul(Wh, xh, 1024)
    assert_close(gpu_matmul(q8, dev(Wh), dev(xh), 1024), ref, bound, "config 1")


@pytest.mark.parametrize("n_tok", [1, 4, 16])
def test_config2_decode_sweep(q8, o, n_tok):
    Wh = inputs.weights(32768, 1024, seed=0)
    xh = inputs.normal((n_tok, 1024), seed=0, p_out=0.01, out_scale=20.0)
    ref, bound = o.matmul(Wh, xh, 32768)
    assert_close(gpu_matmul(q8, dev(Wh), dev(xh), 32768), ref, bound, f"config 2 n={n_tok}")


def _sampled_check(q8, o, W, x, in_dim, out_dim, n_tok, n_sample=3000, full_tokens=(0,), seed=0):
    Wd, xd = dev(W), dev(x)
    got = gpu_matmul(q8, Wd, xd, out_dim)
    xq = o.quantize(x)
    g = np.random.default_rng(seed)
    tok = np.concatenate([g.integers(0, n_tok, n_sample)] + [np.full(out_dim, t) for t in full_tokens])
    row = np.concatenate([g.integers(0, out_dim, n_sample)] + [np.arange(out_dim) for _ in full_tokens])
    ref, bound = o.matmul_sample(W, xq, in_dim, out_dim, n_tok, tok, row)
    assert_close(got[tok, row], ref, bound, f"sampled {in_dim}x{out_dim}x{n_tok}")
    return got


@pytest.mark.parametrize("in_dim,out_dim", [(32768, 1024), (4096, 2048), (2048, 4096)])
def test_config3_prefill(q8, o, in_dim, out_dim):
    W = inputs.weights(out_dim, in_dim, seed=1)
    x = inputs.normal((512, in_dim), seed=1)
    _sampled_check(q8, o, W, x, in_dim, out_dim, 512, full_tokens=(0, 511))


@pytest.mark.parametrize("in_dim,out_dim", [(4096, 1024), (1024, 32768), (32768, 1024), (1024, 4096)])
def test_config5_dense_layer_slice(q8, o, in_dim, out_dim):
    W = inputs.weights(out_dim, in_dim, seed=2)
    x = inputs.normal((4096, in_dim), seed=2)
    _sampled_check(q8, o, W, x, in_dim, out_dim, 4096, full_tokens=(4095,))


# ------------------------------------------------------------------ routed experts
def gpu_moe(q8, Wd, n_exp, stride, ids, x, x_per_pair, out_dim):
    n_tok, k = ids.shape
    buf = poisoned(n_tok * k * out_dim)
    rc = q8.q8_moe_matmul(buf, Wd, n_exp, stride, dev(ids), k, x.shape[1], out_dim, dev(x), int(x_per_pair), n_tok)
    assert rc == 0, q8.q8_strerror(rc)
    return buf, n_tok * k * out_dim


def test_moe_small_every_output(q8, o):
    n_exp, in_dim, out_dim, n_tok, k = 12, 512, 72, 37, 3
    W = inputs.weights(n_exp * out_dim, in_dim, seed=21)
    stride = out_dim * in_dim // QK * QB
    ids = inputs.route_zipf(n_tok, k, n_exp, seed=22)
    for per_pair in (0, 1):
        x = inputs.normal((n_tok * k if per_pair else n_tok, in_dim), seed=23 + per_pair)
        ref, bound, flag = o.moe(W, n_exp, stride, ids, in_dim, out_dim, o.quantize(x), per_pair, n_tok)
        buf, n = gpu_moe(q8, dev(W), n_exp, stride, ids, x, per_pair, out_dim)
        assert q8.q8_last_error() == 0 and flag == 0
        assert_close(fetch(buf, n, ref.shape), ref, bound, f"moe per_pair={per_pair}")


def test_moe_ragged_in_dim_slow_path(q8, o):
    n_exp, in_dim, out_dim, n_tok, k = 5, 96, 20, 9, 2
    W = inputs.weights(n_exp * out_dim, in_dim, seed=31)
    stride = (out_dim * in_dim // QK * QB + 15) // 16 * 16
    Wpad = np.zeros(n_exp * stride, np.uint8)
    for e in range(n_exp):
        Wpad[e * stride:e * stride + out_dim * 3 * QB] = W[e * out_dim:(e + 1) * out_dim].reshape(-1)
    ids = inputs.route_uniform(n_tok, k, n_exp, seed=32)
    x = inputs.normal((n_tok, in_dim), seed=33)
    ref, bound, _ = o.moe(Wpad, n_exp, stride, ids, in_dim, out_dim, o.quantize(x), 0, n_tok)
    buf, n = gpu_moe(q8, dev(Wpad), n_exp, stride, ids, x, 0, out_dim)
    assert q8.q8_last_error() == 0
    assert_close(fetch(buf, n, ref.shape), ref, bound, "moe ragged")


def test_moe_bad_ids_zero_rows_and_flag(q8, o):
    n_exp, in_dim, out_dim, n_tok, k = 6, 256, 40, 10, 2
    W = inputs.weights(n_exp * out_dim, in_dim, seed=41)
    stride = out_dim * in_dim // QK * QB
    ids = inputs.route_uniform(n_tok, k, n_exp, seed=42)
    ids[3, 1] = -1
    ids[7, 0] = 6
    x = inputs.normal((n_tok, in_dim), seed=43)
    ref, bound, flag = o.moe(W, n_exp, stride, ids, in_dim, out_dim, o.quantize(x), 0, n_tok)
    assert flag == 1
    buf, n = gpu_moe(q8, dev(W), n_exp, stride, ids, x, 0, out_dim)
    assert q8.q8_last_error() == q8.Q8_ERANGE
    assert q8.q8_last_error() == 0   # cleared
    got = fetch(buf, n, ref.shape)
    assert np.all(got[3 * k + 1] == 0) and np.all(got[7 * k + 0] == 0)
    assert_close(got, ref, bound, "moe bad ids")


def test_moe_k1_identity_equals_dense(q8, o):
    """k = 1, token e -> expert e: every routed row equals the dense product of that expert,
    within the tolerance (the two calls may sum blocks in different fp32 orders)."""
    n_exp, in_dim, out_dim = 4, 1024, 96
    W = inputs.weights(n_exp * out_dim, in_dim, seed=51)
    stride = out_dim * in_dim // QK * QB
    x = inputs.normal((n_exp, in_dim), seed=52)
    ids = np.arange(n_exp, dtype=np.int32).reshape(n_exp, 1)
    Wd = dev(W)
    moe = q8.moe_matmul(Wd, n_exp, stride, dev(ids), dev(x), False, out_dim).cpu().numpy()
    for e in range(n_exp):
        dense = q8.matmul(Wd[e * out_dim:(e + 1) * out_dim], dev(x[e:e + 1]), out_dim).cpu().numpy()
        ref, bound = o.matmul(W[e * out_dim:(e + 1) * out_dim], x[e:e + 1], out_dim)
        assert_close(moe[e:e + 1], ref, bound, "moe k=1")
        assert_close(dense, ref, bound, "dense")
        assert np.all(np.abs(moe[e:e + 1] - dense) <= 2 * oracle.tolerance(bound))


def test_moe_deterministic(q8):
    n_exp, in_dim, out_dim, n_tok, k = 16, 1024, 256, 40, 4
    W = dev(inputs.weights(n_exp * out_dim, in_dim, seed=53))
    stride = out_dim * in_dim // QK * QB
    ids = dev(inputs.route_zipf(n_tok, k, n_exp, seed=54))
    x = dev(inputs.normal((n_tok, in_dim), seed=55))
    a = q8.moe_matmul(W, n_exp, stride, ids, x, False, out_dim)
    for _ in range(3):
        assert torch.equal(a, q8.moe_matmul(W, n_exp, stride, ids, x, False, out_dim))


def _moe_weights(n_exp, out_dim, in_dim, seed):
    return inputs.weights(n_exp * out_dim, in_dim, seed=seed)


def test_config4_routed_moe_gate_and_down(q8, o):
    n_exp, n_tok, k = 256, 64, 6
    ids = inputs.route_uniform(n_tok, k, n_exp, seed=0)
    # gate/up: experts [2048 x 4096], x per token
    W = _moe_weights(n_exp, 2048, 4096, seed=0)
    stride = 2048 * 128 * QB
    x = inputs.normal((n_tok, 4096), seed=0)
    ref, bound, flag = o.moe(W, n_exp, stride, ids, 4096, 2048, o.quantize(x), 0, n_tok)
    buf, n = gpu_moe(q8, dev(W), n_exp, stride, ids, x, 0, 2048)
    assert q8.q8_last_error() == 0 and flag == 0
    assert_close(fetch(buf, n, ref.shape), ref, bound, "config 4 gate")
    del W, buf
    # down: experts [4096 x 2048], x per pair
    W = _moe_weights(n_exp, 4096, 2048, seed=1)
    stride = 4096 * 64 * QB
    x = inputs.normal((n_tok * k, 2048), seed=1)
    ref, bound, flag = o.moe(W, n_exp, stride, ids, 2048, 4096, o.quantize(x), 1, n_tok)
    buf, n = gpu_moe(q8, dev(W), n_exp, stride, ids, x, 1, 4096)
    assert q8.q8_last_error() == 0
    assert_close(fetch(buf, n, ref.shape), ref, bound, "config 4 down")


def test_config5_zipf_moe_sampled(q8, o):
    n_exp, n_tok, k, in_dim, out_dim = 256, 4096, 6, 4096, 2048
    ids = inputs.route_zipf(n_tok, k, n_exp, s=1.1, seed=0)
    W = _moe_weights(n_exp, out_dim, in_dim, seed=2)
    stride = out_dim * (in_dim // QK) * QB
    x = inputs.normal((n_tok, in_dim), seed=3)
    buf, n = gpu_moe(q8, dev(W), n_exp, stride, ids, x, 0, out_dim)
    assert q8.q8_last_error() == 0
    got = fetch(buf, n, (n_tok * k, out_dim))
    g = np.random.default_rng(5)
    counts = np.bincount(ids.reshape(-1), minlength=n_exp)
    hot = int(np.argmax(counts))
    cold_pairs = np.flatnonzero(np.isin(ids.reshape(-1), np.flatnonzero(counts == counts[counts > 0].min())))[:2]
    hot_pair = int(np.flatnonzero(ids.reshape(-1) == hot)[-1])
    pair = np.concatenate([g.integers(0, n_tok * k, 3000), np.full(out_dim, hot_pair),
                           np.repeat(cold_pairs, out_dim)])
    row = np.concatenate([g.integers(0, out_dim, 3000), np.arange(out_dim), np.tile(np.arange(out_dim), len(cold_pairs))])
    ref, bound, flag = o.moe_sample(W, n_exp, stride, ids, in_dim, out_dim, o.quantize(x), 0, n_tok, pair, row)
    assert flag == 0
    assert_close(got[pair, row], ref, bound, "config 5 moe")
    assert not np.any(np.isnan(got)), "some routed output row was never written"


def test_config5_zipf_moe_down_sampled(q8, o):
    """The long-prefill slice's routed down projection at its real size: one input row per
    pair (24576 pairs, Zipf(1.1) top-6 over 256 experts of 4096 x 2048), on the grouped
    tcgen05 GEMM and the GEMV classes.  Random outputs plus whole rows of the hottest
    expert's last pair and the coldest experts' first pairs are checked."""
    n_exp, n_tok, k, in_dim, out_dim = 256, 4096, 6, 2048, 4096
    ids = inputs.route_zipf(n_tok, k, n_exp, s=1.1, seed=0)
    W = _moe_weights(n_exp, out_dim, in_dim, seed=4)
    stride = out_dim * (in_dim // QK) * QB
    x = inputs.normal((n_tok * k, in_dim), seed=5)
    buf, n = gpu_moe(q8, dev(W), n_exp, stride, ids, x, 1, out_dim)
    assert q8.q8_last_error() == 0
    got = fetch(buf, n, (n_tok * k, out_dim))
    assert not np.any(np.isnan(got)), "some routed output row was never written"
    flat = ids.reshape(-1)
    counts = np.bincount(flat, minlength=n_exp)
    assert counts.max() > 1000 and counts[counts > 0].min() <= 16   # tensor-core and GEMV classes
    hot_pair = int(np.flatnonzero(flat == int(np.argmax(counts)))[-1])
    cold = np.flatnonzero(counts == counts[counts > 0].min())
    cold_pairs = [int(np.flatnonzero(flat == e)[0]) for e in cold[:2]]
    mid_e = int(np.flatnonzero((counts > 16) & (counts < 128))[0])           # a short tensor-core group
    mid_pair = int(np.flatnonzero(flat == mid_e)[-1])
    whole = [hot_pair, mid_pair] + cold_pairs
    g = np.random.default_rng(6)
    pair = np.concatenate([g.integers(0, n_tok * k, 4000), np.repeat(whole, out_dim)])
    row = np.concatenate([g.integers(0, out_dim, 4000), np.tile(np.arange(out_dim), len(whole))])
    ref, bound, flag = o.moe_sample(W, n_exp, stride, ids, in_dim, out_dim, o.quantize(x), 1, n_tok, pair, row)
    assert flag == 0
    assert_close(got[pair, row], ref, bound, "config 5 routed down")


def _ids_with_counts(counts, k, seed):
    """int32 [n_pairs / k, k]: expert e appears counts[e] times, in a seeded random order."""
    flat = np.repeat(np.arange(len(counts), dtype=np.int32), counts)
    assert flat.size % k == 0
    flat = np.random.default_rng(seed).permutation(flat).astype(np.int32)
    return flat.reshape(-1, k)


# Groups around the class edges: 1-8 rows run on the GEMV in one 8-token tile,
# 9-16 in 16-token groups, larger groups on the grouped tcgen05 GEMM, whose
# last tile of a group is 32, 64 or 128 tokens wide: 17 / 32 / 33 / 64 / 65
# straddle those widths, 127 / 128 / 129 one full tile, 300 spans three.
TC_COUNTS = [65, 127, 128, 129, 200, 300, 1, 2, 3, 5, 8, 9, 16, 17, 33, 64, 32, 1]


@pytest.mark.parametrize("in_dim,out_dim", [(256, 200), (2048, 136)])
def test_moe_tensor_core_class_every_output(q8, o, in_dim, out_dim):
    """Batches of >= 1024 pairs send groups of more than 16 rows to the grouped tcgen05
    GEMM; every output of every class is checked, and a second call must agree bit for bit."""
    n_exp, k = len(TC_COUNTS), 3
    ids = _ids_with_counts(TC_COUNTS, k, seed=81)
    n_tok = ids.shape[0]
    assert n_tok * k >= 1024
    W = inputs.weights(n_exp * out_dim, in_dim, seed=82)
    stride = out_dim * in_dim // QK * QB
    Wd = dev(W)
    for per_pair in (0, 1):
        x = inputs.normal((n_tok * k if per_pair else n_tok, in_dim), seed=83 + per_pair, p_out=0.01)
        ref, bound, flag = o.moe(W, n_exp, stride, ids, in_dim, out_dim, o.quantize(x), per_pair, n_tok)
        assert flag == 0
        buf, n = gpu_moe(q8, Wd, n_exp, stride, ids, x, per_pair, out_dim)
        assert q8.q8_last_error() == 0
        got = fetch(buf, n, ref.shape)
        assert_close(got, ref, bound, f"moe tensor-core class per_pair={per_pair}")
        buf2, _ = gpu_moe(q8, Wd, n_exp, stride, ids, x, per_pair, out_dim)
        assert np.array_equal(fetch(buf2, n, ref.shape), got)


def test_moe_tensor_core_class_empty(q8, o):
    """A batch large enough for the tensor-core class, but no group of more than 16 rows."""
    n_exp, n_tok, k, in_dim, out_dim = 256, 512, 2, 256, 72
    ids = inputs.route_uniform(n_tok, k, n_exp, seed=84)
    assert np.bincount(ids.reshape(-1), minlength=n_exp).max() <= 16
    W = inputs.weights(n_exp * out_dim, in_dim, seed=85)
    stride = out_dim * in_dim // QK * QB
    x = inputs.normal((n_tok, in_dim), seed=86)
    ref, bound, _ = o.moe(W, n_exp, stride, ids, in_dim, out_dim, o.quantize(x), 0, n_tok)
    buf, n = gpu_moe(q8, dev(W), n_exp, stride, ids, x, 0, out_dim)
    assert q8.q8_last_error() == 0
    assert_close(fetch(buf, n, ref.shape), ref, bound, "moe without tensor-core groups")


def test_moe_many_experts_every_output(q8, o):
    """12000 experts: the routing plan's shared-memory arrays (96 KB) need the opt-in
    limit; Zipf routing over 1600 pairs gives tensor-core, 16-token and 8-token groups."""
    n_exp, n_tok, k, in_dim, out_dim = 12000, 200, 8, 256, 24
    ids = inputs.route_zipf(n_tok, k, n_exp, s=1.1, seed=91)
    counts = np.bincount(ids.reshape(-1), minlength=n_exp)
    assert counts.max() > 16 and np.any((counts > 8) & (counts <= 16)) and np.any((counts > 0) & (counts <= 8))
    W = inputs.weights(n_exp * out_dim, in_dim, seed=92)
    stride = out_dim * in_dim // QK * QB
    x = inputs.normal((n_tok, in_dim), seed=93)
    ref, bound, flag = o.moe(W, n_exp, stride, ids, in_dim, out_dim, o.quantize(x), 0, n_tok)
    assert flag == 0
    buf, n = gpu_moe(q8, dev(W), n_exp, stride, ids, x, 0, out_dim)
    assert q8.q8_last_error() == 0
    assert_close(fetch(buf, n, ref.shape), ref, bound, "moe 12000 experts")


def test_moe_tensor_core_large_experts_sampled(q8, o):
    """Twenty experts of 4096 x 16384 with 70 rows each, all on the grouped tcgen05 GEMM
    (32 weight tiles per expert, 64 raw copies of 8 blocks per tile).  Whole output rows of
    six experts are checked, plus random elements."""
    n_exp, k, in_dim, out_dim, per = 20, 1, 16384, 4096, 70
    ids = _ids_with_counts([per] * n_exp, k, seed=87)
    n_tok = ids.shape[0]
    W = inputs.weights(n_exp * out_dim, in_dim, seed=88)
    stride = out_dim * (in_dim // QK) * QB
    x = inputs.normal((n_tok, in_dim), seed=89)
    buf, n = gpu_moe(q8, dev(W), n_exp, stride, ids, x, 0, out_dim)
    assert q8.q8_last_error() == 0
    got = fetch(buf, n, (n_tok * k, out_dim))
    flat = ids.reshape(-1)
    whole = [int(np.flatnonzero(flat == e)[j]) for e, j in ((0, 0), (15, -1), (16, 0), (17, 5), (18, 33), (19, -1))]
    g = np.random.default_rng(90)
    pair = np.concatenate([g.integers(0, n_tok * k, 2000), np.repeat(whole, out_dim)])
    row = np.concatenate([g.integers(0, out_dim, 2000), np.tile(np.arange(out_dim), len(whole))])
    ref, bound, flag = o.moe_sample(W, n_exp, stride, ids, in_dim, out_dim, o.quantize(x), 0, n_tok, pair, row)
    assert flag == 0
    assert_close(got[pair, row], ref, bound, "moe large experts")
    assert not np.any(np.isnan(got)), "some routed output row was never written"


# ------------------------------------------------------------------ repack
def test_repack_layout_and_parity(q8, o):
    in_dim, out_dim, n_tok = 1024, 200, 13
    Wh = inputs.weights(out_dim, in_dim, seed=61)
    Wp = q8.repack(dev(Wh), in_dim, out_dim).cpu().numpy()
    blk = Wh.reshape(out_dim, -1, QB)
    assert np.array_equal(Wp[:out_dim * in_dim].reshape(out_dim, -1, QK), blk[..., 2:])
    assert np.array_equal(Wp[out_dim * in_dim:].reshape(out_dim, -1, 2), blk[..., :2])
    xh = inputs.normal((n_tok, in_dim), seed=62)
    ref, bound = o.matmul(Wh, xh, out_dim)
    got = q8.matmul_packed(dev(Wp), dev(xh), out_dim).cpu().numpy()
    assert_close(got, ref, bound, "packed")


@pytest.mark.parametrize("in_dim,out_dim", [(1024, 200), (2112, 130), (64, 7), (4096, 1024)])
def test_repack_tensor_core_layout_and_parity(q8, o, in_dim, out_dim):
    """The tcgen05 GEMM's weight operand built once: fp16 quants (exact integers) in [m_ld][in_dim] and
    the binary16 scales as fp32 in [in_dim/32][m_ld], padding rows zero.  Its products match the oracle
    for few and many tokens, and above 2048 tokens are the bits of q8_matmul (which then expands the
    weights into the same layout per call)."""
    Wh = inputs.weights(out_dim, in_dim, seed=63)
    W = dev(Wh)
    Wp = q8.repack(W, in_dim, out_dim, q8.Q8_LAYOUT_TC)
    nb, m_ld = in_dim // QK, (out_dim + 127) // 128 * 128
    h = Wp.cpu().numpy()
    q16 = h[:m_ld * in_dim * 2].view(np.float16).reshape(m_ld, nb, QK)
    dT = h[m_ld * in_dim * 2:].view(np.float32).reshape(nb, m_ld)
    blk = Wh.reshape(out_dim, nb, QB)
    assert np.array_equal(q16[:out_dim].astype(np.int64), blk[..., 2:].view(np.int8).astype(np.int64))
    assert np.array_equal(dT[:, :out_dim].T, blk[..., :2].copy().view(np.float16).reshape(out_dim, nb).astype(np.float32))
    assert not np.any(q16[out_dim:]) and not np.any(dT[:, out_dim:])
    for n_tok in (1, 16, 40, 2100):
        xh = inputs.normal((n_tok, in_dim), seed=64 + n_tok, p_out=0.01)
        x = dev(xh)
        got = q8.matmul_packed(Wp, x, out_dim, q8.Q8_LAYOUT_TC)
        if n_tok <= 40:
            ref, bound = o.matmul(Wh, xh, out_dim)
            assert_close(got.cpu().numpy(), ref, bound, f"tc-packed {in_dim}x{out_dim}x{n_tok}")
        else:
            assert torch.equal(got, q8.matmul(W, x, out_dim))


# ------------------------------------------------------------------ host-buffer entry point
def _host_call(q8, W, xh, out_dim, pinned):
    n_tok, in_dim = xh.shape
    x_host = torch.from_numpy(np.ascontiguousarray(xh))
    out_host = torch.full((n_tok * out_dim + GUARD,), float("nan"), dtype=torch.float32)
    if pinned:
        x_host, out_host = x_host.pin_memory(), out_host.pin_memory()
    rc = q8.q8_matmul_host(out_host, W, in_dim, out_dim, x_host, n_tok)
    assert rc == 0, f"{q8.q8_strerror(rc)} {q8.q8_last_cuda_error()}"
    assert q8.q8_last_error() == 0                      # synchronises the stream
    h = out_host.numpy()
    assert np.all(np.isnan(h[n_tok * out_dim:])), "guard band after the host output was written"
    return h[:n_tok * out_dim].reshape(n_tok, out_dim)


@pytest.mark.parametrize("n_tok,in_dim,out_dim", [(1, 1024, 300), (4, 1024, 300), (16, 1024, 3000),
                                                   (40, 2048, 300), (700, 1024, 200)])
@pytest.mark.parametrize("pinned", [True, False])
def test_matmul_host_matches_matmul_bitwise(q8, n_tok, in_dim, out_dim, pinned):
    """Host x and out around the same kernels: the bits of q8_matmul, for the
    GEMV (from the quantiser's planes when x is mapped host memory, fused otherwise:
    the same quantised values either way), and both tensor-core variants."""
    W = dev(inputs.weights(out_dim, in_dim, seed=91))
    xh = inputs.normal((n_tok, in_dim), seed=92, p_out=0.01)
    ref = q8.matmul(W, dev(xh), out_dim).cpu().numpy()
    got = _host_call(q8, W, xh, out_dim, pinned)
    assert np.array_equal(got.view(np.int32), ref.view(np.int32))


def test_matmul_host_oracle_and_repeat(q8, o):
    """Against the oracle, and back-to-back calls of different sizes on one stream
    (each call's copy-in waits for the previous call's kernels)."""
    Wh = inputs.weights(500, 2048, seed=93)
    W = dev(Wh)
    for n_tok in (5, 16, 1, 33):
        xh = inputs.normal((n_tok, 2048), seed=94 + n_tok)
        ref, bound = o.matmul(Wh, xh, 500)
        assert_close(_host_call(q8, W, xh, 500, True), ref, bound, f"host {n_tok}")


@pytest.mark.parametrize("n_tok", [4, 16])
def test_matmul_host_two_items_per_cta(q8, o, n_tok):
    """out 32768 with the result in host memory: every CTA takes two items of six or
    seven 16-row sub-items (two warps a sub-item, partial sums added in slice order),
    so the first item's results cross the host link while the second item's weights
    stream.  Every output against the oracle."""
    in_dim, out_dim = 1024, 32768
    Wh = inputs.weights(out_dim, in_dim, seed=97)
    W = dev(Wh)
    xh = inputs.normal((n_tok, in_dim), seed=98 + n_tok, p_out=0.01)
    ref, bound = o.matmul(Wh, xh, out_dim)
    assert_close(_host_call(q8, W, xh, out_dim, True), ref, bound, f"host out {out_dim} x {n_tok}")


def test_matmul_host_errors(q8):
    W = dev(inputs.weights(64, 256, seed=95))
    x_host = torch.from_numpy(inputs.normal((3, 256), seed=96))
    out_host = torch.empty((3, 64), dtype=torch.float32)
    assert q8.q8_matmul_host(out_host, W, 256, 64, None, 3) == q8.Q8_EINVAL
    assert q8.q8_matmul_host(None, W, 256, 64, x_host, 3) == q8.Q8_EINVAL
    assert q8.q8_matmul_host(out_host, W, 250, 64, x_host, 3) == q8.Q8_EINVAL
    assert q8.q8_matmul_host(out_host, W.data_ptr() + 1, 256, 64, x_host, 3) == q8.Q8_EALIGN
    assert q8.q8_matmul_host(out_host, W, 256, 64, x_host, 0) == 0
    # the staging buffer is library scratch: freed by q8_release, and an allocation
    # failure enqueues nothing and leaves the next call working
    q8.q8_release()
    assert q8.q8_scratch_bytes() == 0
    q8.q8_debug_fail_next_alloc(1)
    assert q8.q8_matmul_host(out_host, W, 256, 64, x_host, 3) == q8.Q8_ENOMEM
    assert q8.q8_matmul_host(out_host, W, 256, 64, x_host, 3) == 0
    assert q8.q8_last_error() == 0
    assert q8.q8_scratch_bytes() > 0
    assert torch.equal(out_host, q8.matmul(W, x_host.to(DEV), 64).cpu())


# ------------------------------------------------------------------ error paths and edges
def test_empty_and_tiny(q8, o):
    W = dev(inputs.weights(3, 32, seed=71))
    x = dev(inputs.normal((1, 32), seed=72))
    out = torch.empty((0, 3), device=DEV)
    assert q8.q8_matmul(out, W, 32, 3, x, 0) == 0
    ref, bound = o.matmul(inputs.weights(3, 32, seed=71), inputs.normal((1, 32), seed=72), 3)
    assert_close(q8.matmul(W, x, 3).cpu().numpy(), ref, bound, "tiny")


def test_scratch_alloc_failure_reports_enomem(q8):
    W = dev(inputs.weights(64, 256, seed=81))
    x = dev(inputs.normal((20, 256), seed=82))
    out = torch.empty((20, 64), device=DEV)
    q8.q8_release()
    assert q8.q8_scratch_bytes() == 0
    # a small decode call quantises inside the GEMV and needs no scratch
    assert q8.q8_matmul(out, W, 256, 64, x, 8) == 0
    assert q8.q8_scratch_bytes() == 0
    # 20 tokens take the tensor-core path, whose operands live in scratch
    q8.q8_debug_fail_next_alloc(1)
    assert q8.q8_matmul(out, W, 256, 64, x, 20) == q8.Q8_ENOMEM
    assert q8.q8_matmul(out, W, 256, 64, x, 20) == 0
    assert q8.q8_scratch_bytes() > 0
    torch.cuda.synchronize()
