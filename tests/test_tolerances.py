"""The agreement rules of the GPU parity tests, tested on the CPU with the oracle
alone (no GPU): each rule must accept differences of the size the kernels' fp32
arithmetic makes, and reject planted mistakes.  Kernel-like results are made by
moving the oracle's own intermediates by fp32-sized amounts and running the rest
of the oracle on them; mistakes are planted in the oracle's inputs or arguments.
"""
import numpy as np
import pytest

import inputs
import oracle
from tests import allowances

QK, QB = 32, 34


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def _ffn_instance(seed=40):
    n_exp, in_dim, mid_dim, out_dim, n_tok, k = 16, 512, 256, 384, 24, 4
    Wg = inputs.weights(n_exp * mid_dim, in_dim, seed=seed).reshape(-1)
    Wu = inputs.weights(n_exp * mid_dim, in_dim, seed=seed + 1).reshape(-1)
    Wd = inputs.weights(n_exp * out_dim, mid_dim, seed=seed + 2).reshape(-1)
    gu, ds = mid_dim * (in_dim // QK) * QB, out_dim * (mid_dim // QK) * QB
    ids = inputs.route_uniform(n_tok, k, n_exp, seed=seed)
    w = np.random.default_rng(seed).random((n_tok, k)).astype(np.float32)
    x = inputs.normal((n_tok, in_dim), seed=seed, p_out=0.01)
    return dict(Wg=Wg, Wu=Wu, Wd=Wd, gu=gu, ds=ds, ids=ids, w=w, x=x, n_exp=n_exp, in_dim=in_dim,
                mid_dim=mid_dim, out_dim=out_dim, n_tok=n_tok, k=k)


def _ffn(o, c, limit, **kw):
    a = {**c, **kw}
    return o.moe_ffn(a["Wg"], a["Wu"], a["Wd"], a["n_exp"], a["gu"], a["ds"], a["ids"], a["w"], a["in_dim"],
                     a["mid_dim"], a["out_dim"], limit, a["x"])


@pytest.mark.parametrize("limit", [10.0, 0.0])
def test_ffn_tolerance_accepts_fp32_scale_differences(o, limit):
    """gate and up moved by 1e-6 relative (ten times the fp32 differences of the GPU's
    sums), then SwiGLU, re-quantisation, down and the weighted sum by the oracle: every
    output stays within oracle.ffn_tolerance, although quants of mid do flip."""
    c = _ffn_instance()
    r = _ffn(o, c, limit)
    tol = oracle.ffn_tolerance(r, c["Wd"], c["ds"], c["ids"], c["w"], c["mid_dim"], c["out_dim"])
    xq = o.quantize(c["x"])
    gate, _, _ = o.moe(c["Wg"], c["n_exp"], c["gu"], c["ids"], c["in_dim"], c["mid_dim"], xq, 0, c["n_tok"])
    up, _, _ = o.moe(c["Wu"], c["n_exp"], c["gu"], c["ids"], c["in_dim"], c["mid_dim"], xq, 0, c["n_tok"])
    flipped = 0
    for trial in range(6):
        g = np.random.default_rng(trial)
        gp = (gate * (1 + 1e-6 * g.standard_normal(gate.shape))).astype(np.float32)
        upp = (up * (1 + 1e-6 * g.standard_normal(up.shape))).astype(np.float32)
        midq = o.quantize(o.swiglu(gp, upp, limit))
        flipped += int(np.sum(midq != r["midq"]))
        y, _, _ = o.moe(c["Wd"], c["n_exp"], c["ds"], c["ids"], c["mid_dim"], c["out_dim"], midq, 1, c["n_tok"])
        out, _ = o.combine(y, c["w"].reshape(-1), c["n_tok"], c["k"])
        assert np.all(np.abs(out - r["out"]) <= tol), trial
    assert flipped > 0, "no quant of mid flipped: the test did not exercise the allowance"


def test_ffn_tolerance_rejects_planted_mistakes(o):
    c = _ffn_instance()
    r = _ffn(o, c, 10.0)
    tol = oracle.ffn_tolerance(r, c["Wd"], c["ds"], c["ids"], c["w"], c["mid_dim"], c["out_dim"])
    frac = lambda bad: np.mean(np.abs(bad["out"] - r["out"]) > tol)
    w0 = c["w"].copy()
    w0[:, 0] = 0.0                                                    # first slot dropped
    assert frac(_ffn(o, c, 10.0, w=w0)) > 0.9
    assert frac(_ffn(o, c, 0.0)) > 0.9                                 # clamp not applied
    assert frac(_ffn(o, c, 10.0, Wg=c["Wu"], Wu=c["Wg"])) > 0.9        # gate and up swapped
    ids = c["ids"].copy()
    ids[:, 1] = (ids[:, 1] + 1) % c["n_exp"]                           # wrong expert in slot 1
    bad = _ffn(o, c, 10.0, ids=ids)
    assert np.mean(np.abs(bad["out"] - r["out"]) > tol) > 0.9


def _rms_case(o, dim, n_tok=8):
    x = inputs.normal((n_tok, dim), seed=dim, p_out=0.01)
    gamma = (1.0 + 0.3 * np.random.default_rng(dim).standard_normal(dim)).astype(np.float32)
    xq_o, y_o = o.rmsnorm_quantize(x, gamma, 1e-6)
    return x, gamma, xq_o, y_o


@pytest.mark.parametrize("dim", [4096, 2080, 96])
def test_rmsnorm_rules_accept_fp32_scale_differences(o, dim):
    """y moved by half the kernel's bound per row (the error of its 1/rms) and by one fp32
    rounding per value, then quantised by the oracle (bit-exact to the kernel's quantiser):
    the rules accept it, although quants flip at ties."""
    _, _, xq_o, y_o = _rms_case(o, dim, n_tok=32)
    r = allowances.rms_rho(dim)
    flipped = 0
    for trial in range(5):
        g = np.random.default_rng(trial)
        row = 1.0 + 0.5 * r * g.uniform(-1, 1, (y_o.shape[0], 1))
        yk = (y_o.astype(np.float64) * row).astype(np.float32)
        xqk = o.quantize(yk)
        flipped += int(np.sum(xqk != xq_o))
        allowances.check_rmsnorm(xqk, yk, xq_o, y_o)
    if dim == 4096:
        assert flipped > 0, "no quant flipped: the test did not exercise the allowance"


def test_rmsnorm_rules_reject_planted_mistakes(o):
    x, gamma, xq_o, y_o = _rms_case(o, 4096)
    for bad in (o.rmsnorm_quantize(x, None, 1e-6),                       # gamma ignored
                o.rmsnorm_quantize(x, gamma, 1.0),                        # eps far too large
                o.rmsnorm_quantize(x * np.float32(1.5), gamma, 1e2)):     # not scale-free
        with pytest.raises(AssertionError):
            allowances.check_rmsnorm(bad[0], bad[1], xq_o, y_o)
    r = allowances.rms_rho(4096)
    yk = (y_o.astype(np.float64) * (1 + 4 * r)).astype(np.float32)         # y beyond its bound
    with pytest.raises(AssertionError):
        allowances.check_rmsnorm(o.quantize(yk), yk, xq_o, y_o)
    nb = 4096 // QK
    d, q = allowances.split_blocks(xq_o, nb)
    d32 = np.abs(y_o.reshape(-1, nb, QK)).max(-1) / np.float32(127.0)
    quo = np.abs(y_o.reshape(-1, nb, QK) / d32[..., None])
    t, b, i = np.unravel_index(np.argmax(np.abs(quo - np.floor(quo) - 0.5)), quo.shape)   # farthest from a tie
    xq_bad = xq_o.copy().reshape(-1, nb, QB)
    qv = int(np.int8(xq_bad[t, b, 2 + i].view(np.int8)))
    xq_bad[t, b, 2 + i] = np.array([qv - 1 if qv > -127 else qv + 1], np.int8).view(np.uint8)[0]
    with pytest.raises(AssertionError):
        allowances.check_rmsnorm(xq_bad.reshape(xq_o.shape), y_o, xq_o, y_o)
    xq_bad = xq_o.copy().reshape(-1, nb, QB)
    hb = int(xq_bad[0, 0, 0]) | (int(xq_bad[0, 0, 1]) << 8)
    hb += 1                                                                  # scale one binary16 step up
    xq_bad[0, 0, 0], xq_bad[0, 0, 1] = hb & 0xFF, hb >> 8
    with pytest.raises(AssertionError):
        allowances.check_rmsnorm(xq_bad.reshape(xq_o.shape), y_o, xq_o, y_o)
