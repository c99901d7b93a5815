"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` instance and raises
AssertionError when the oracle disagrees with

* a library routine (numpy's IEEE binary16 conversion),
* a closed form (exactly representable blocks round-trip, hand-built ties,
  one-hot products, power-of-two scaling, the integer matmul when every scale
  is 1),
* an invariant (sign symmetry, |x/d - q| <= 1/2, all-zero blocks give 0,
  max |q| = 127 at the block maximum), or
* brute force in exact rational arithmetic on tiny inputs, within the rounding
  bound of an fp32 sum.

The same functions run against planted-mistake copies of the oracle
(tests/test_oracle_mutants.py) to show that each plausible mistake fails at
least one pin.  The formulas come from the ds4 pages: the Q8_K quantiser
(model-architecture page, quantisation section 1), the Q8_0 matmul
(GPU code walkthrough, trace 3) and the fixed-point block dot product
(quantisation section 4).
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np

QK = 32
QB = 34
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- helpers
def make_blocks(d_bits: np.ndarray, q: np.ndarray) -> np.ndarray:
    """Assemble raw 34-byte blocks from fp16 bit patterns [..., nb] and int8 q [..., nb, 32]."""
    d_bits = np.asarray(d_bits, dtype=np.uint16)
    q = np.asarray(q, dtype=np.int8)
    lead = d_bits.shape
    out = np.empty(lead + (QB,), dtype=np.uint8)
    out[..., 0] = (d_bits & 0xFF).astype(np.uint8)
    out[..., 1] = (d_bits >> 8).astype(np.uint8)
    out[..., 2:] = q.view(np.uint8)
    return out.reshape(lead[:-1] + (lead[-1] * QB,))


def split_blocks(raw: np.ndarray, nb: int):
    """raw [..., nb*34] -> (d_bits uint16 [..., nb], q int8 [..., nb, 32])."""
    r = np.asarray(raw, dtype=np.uint8).reshape(raw.shape[:-1] + (nb, QB))
    d = r[..., 0].astype(np.uint16) | (r[..., 1].astype(np.uint16) << 8)
    q = r[..., 2:].copy().view(np.int8)
    return d, q


def f16_exact(bits) -> Fraction:
    """Exact rational value of a finite binary16 bit pattern (from the format's definition)."""
    bits = int(bits)
    s = -1 if bits & 0x8000 else 1
    e = (bits >> 10) & 0x1F
    f = bits & 0x3FF
    assert e != 31
    if e == 0:
        return s * Fraction(f, 1 << 24)
    return s * Fraction(1024 + f, 1 << 10) * (Fraction(2) ** (e - 15))


def exact_matmul(W, xq, in_dim, out_dim, n_tok):
    """Exact rationals: out[t][o] = sum_b d_w d_x sum_i q_w q_x; also sum_b |.|."""
    nb = in_dim // QK
    dw, qw = split_blocks(W.reshape(out_dim, -1), nb)
    dx, qx = split_blocks(xq.reshape(n_tok, -1), nb)
    isum = np.einsum("obi,tbi->tob", qw.astype(np.int64), qx.astype(np.int64))
    vals = np.empty((n_tok, out_dim), dtype=object)
    bnds = np.empty((n_tok, out_dim), dtype=object)
    for t in range(n_tok):
        for o in range(out_dim):
            acc = Fraction(0)
            bnd = Fraction(0)
            for b in range(nb):
                c = f16_exact(dw[o, b]) * f16_exact(dx[t, b]) * int(isum[t, o, b])
                acc += c
                bnd += abs(c)
            vals[t, o] = acc
            bnds[t, o] = bnd
    return vals, bnds


def rng(seed):
    return np.random.default_rng(seed)


def random_f16_normal_bits(g, n, lo_exp=-14, hi_exp=4):
    """Random positive normal binary16 patterns with unbiased exponent in [lo_exp, hi_exp]."""
    e = g.integers(lo_exp + 15, hi_exp + 16, size=n)
    f = g.integers(0, 1024, size=n)
    return ((e << 10) | f).astype(np.uint16)


# ---------------------------------------------------------------- binary16 pins
def pin_f16_from_f32_matches_library(o):
    """f32 -> f16 (round to nearest even, subnormals, overflow) equals numpy's conversion."""
    g = rng(1)
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24,
            2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -26, 3 * 2.0 ** -26, 2.0 ** -14,
            2.0 ** -14 * (1 - 2 ** -12), 1e-40, 6.1e-5, 5.96e-8, 1 + 2 ** -11, 1 + 3 * 2 ** -11,
            0.1, 1 / 3, 127.0, 0.0078125]
    # exact ties between neighbouring binary16 values (normal and subnormal)
    h = random_f16_normal_bits(g, 500, -14, 14).astype(np.float32)
    base = np.frombuffer(random_f16_normal_bits(g, 500, -14, 14).tobytes(), dtype=np.float16)
    up = np.nextafter(base, np.float16(np.inf))
    ties = (base.astype(np.float64) + up.astype(np.float64)) / 2
    sub = np.arange(0, 1024, dtype=np.float64) * 2.0 ** -24 + 2.0 ** -25
    wide = g.standard_normal(4000) * np.exp(g.uniform(-20, 12, size=4000))
    allv = np.concatenate([np.array(vals), h, ties, -ties, sub, -sub, wide]).astype(np.float32)
    for v in allv:
        with np.errstate(over="ignore"):
            want = int(np.float32(v).astype(np.float16).view(np.uint16))
        got = o.f32_to_f16(float(v))
        assert got == want, f"f32_to_f16({v!r}) = {got:#06x}, numpy {want:#06x}"


def pin_f16_to_f32_matches_library(o):
    """f16 -> f32 equals numpy for every finite and infinite pattern."""
    for bits in range(0, 1 << 16, 7):
        ref = np.array([bits], dtype=np.uint16).view(np.float16)[0]
        got = o.f16_to_f32(bits)
        if np.isnan(ref):
            assert np.isnan(got), bits
        else:
            assert got == float(ref), f"f16_to_f32({bits:#06x}) = {got!r}, numpy {float(ref)!r}"
    for bits in (0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0x7C00, 0x8001, 0xFC00):
        assert o.f16_to_f32(bits) == float(np.array([bits], np.uint16).view(np.float16)[0])


# ---------------------------------------------------------------- quantiser pins
def pin_quantize_zero_block(o):
    """An all-zero block stores d = +0 and q = 0 (also -0.0 inputs)."""
    x = np.zeros((2, 64), dtype=np.float32)
    x[1, :32] = -0.0
    x[1, 32:] = np.linspace(-1, 1, 32)
    xq = o.quantize(x)
    assert np.all(xq[0] == 0)
    assert np.all(xq[1, :QB] == 0)
    assert np.any(xq[1, QB:] != 0)


def pin_quantize_roundtrip_exact(o):
    """x = d*k with d an fp16 value and max|k| = 127 quantises to exactly (d, k)."""
    g = rng(2)
    nb = 24
    d_bits = random_f16_normal_bits(g, nb, -14, 3)
    k = g.integers(-127, 128, size=(nb, QK))
    j = g.integers(0, QK, size=nb)
    k[np.arange(nb), j] = np.where(g.random(nb) < 0.5, 127, -127)
    d = np.frombuffer(d_bits.tobytes(), dtype=np.float16).astype(np.float32)
    x = (d[:, None] * k).astype(np.float32).reshape(1, nb * QK)
    assert np.all(x.astype(np.float64) == d.astype(np.float64)[:, None].repeat(QK, 1).reshape(1, -1) * k.reshape(1, -1))
    xq = o.quantize(x)
    got_d, got_q = split_blocks(xq, nb)
    assert np.array_equal(got_d[0], d_bits), "scale does not round-trip"
    assert np.array_equal(got_q[0], k.astype(np.int8)), "quants do not round-trip"


def pin_quantize_ties_away_from_zero(o):
    """x/d = m + 1/2 exactly rounds away from zero (C roundf), for many scales."""
    g = rng(3)
    nb = 40
    d_bits = random_f16_normal_bits(g, nb, -12, 2)
    d = np.frombuffer(d_bits.tobytes(), dtype=np.float16).astype(np.float64)
    m = g.integers(0, 126, size=(nb, QK)).astype(np.float64)
    sgn = np.where(g.random((nb, QK)) < 0.5, -1.0, 1.0)
    v = sgn * (m + 0.5)
    v[:, 0] = 127.0
    x = (d[:, None] * v).astype(np.float32)
    assert np.all(x.astype(np.float64) == d[:, None] * v)
    xq = o.quantize(x.reshape(1, -1))
    got_d, got_q = split_blocks(xq, nb)
    assert np.array_equal(got_d[0], d_bits)
    want = (sgn * (m + 1)).astype(np.int64)
    want[:, 0] = 127
    assert np.array_equal(got_q[0].astype(np.int64), want), "ties must round away from zero"


def pin_quantize_invariants(o):
    """Random blocks: sign symmetry, |x/d - q| <= 1/2, max|q| = 127 at the block maximum,
    stored d is the nearest binary16 of the fp32 scale amax/127 (numpy conversion)."""
    g = rng(4)
    n_tok, in_dim = 3, 32 * 17
    x = (g.standard_normal((n_tok, in_dim)) * np.exp(g.uniform(-6, 3, size=(n_tok, 1)))).astype(np.float32)
    x[0, 5] *= 20
    nb = in_dim // QK
    xq = o.quantize(x)
    d_bits, q = split_blocks(xq, nb)
    xb = x.reshape(n_tok, nb, QK)
    amax = np.abs(xb).max(axis=2)
    d32 = (amax / np.float32(127)).astype(np.float32)
    assert np.array_equal(d_bits, d32.astype(np.float16).view(np.uint16)), "stored d != fp16(amax/127)"
    ratio = xb.astype(np.float64) / d32.astype(np.float64)[..., None]
    assert np.all(np.abs(ratio - q) <= 0.5 + 1e-6), "quant not nearest"
    assert np.all(np.abs(q.astype(np.int64)).max(axis=2) == 127)
    arg = np.abs(xb).argmax(axis=2)
    assert np.all(np.abs(np.take_along_axis(q.astype(np.int64), arg[..., None], 2)) == 127)
    xq_neg = o.quantize(-x)
    d2, q2 = split_blocks(xq_neg, nb)
    assert np.array_equal(d2, d_bits) and np.array_equal(q2.astype(np.int64), -q.astype(np.int64))


def pin_quantize_subnormal_scale(o):
    """Scales in the binary16 subnormal range are kept (rounded to nearest), not flushed."""
    g = rng(5)
    amax = np.float32(127) * np.float32(2.0 ** -20)  # d = 2^-20, a binary16 subnormal
    x = (g.uniform(-1, 1, size=(1, 64)) * amax).astype(np.float32)
    x[0, 3] = amax
    x[0, 40] = -amax * np.float32(0.37)
    x[0, 33] = -np.float32(127) * np.float32(3.3e-7)
    xq = o.quantize(x)
    d_bits, q = split_blocks(xq, 2)
    amaxes = np.abs(x.reshape(2, 32)).max(axis=1)
    want = (amaxes / np.float32(127)).astype(np.float32).astype(np.float16).view(np.uint16)
    assert np.array_equal(d_bits[0], want)
    assert d_bits[0, 0] == 0x0010 and d_bits[0, 1] < 0x0400


def pin_quantize_golden(o):
    """Hand-derived worked examples (tests/golden/quantize_worked.json)."""
    with open(os.path.join(GOLDEN, "quantize_worked.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        x = np.array(c["x"], dtype=np.float32).reshape(1, -1)
        xq = o.quantize(x)
        d_bits, q = split_blocks(xq, 1)
        assert int(d_bits[0, 0]) == int(c["d_bits"], 16), c["name"]
        assert list(q[0, 0].astype(int)) == c["q"], c["name"]


# ---------------------------------------------------------------- dot / matmul pins
def _rand_weights(g, rows, in_dim, lo_exp=-10, hi_exp=-7):
    nb = in_dim // QK
    d = random_f16_normal_bits(g, rows * nb, lo_exp, hi_exp).reshape(rows, nb)
    q = g.integers(-127, 128, size=(rows, nb, QK))
    return make_blocks(d, q)


def _rand_acts(g, n_tok, in_dim):
    nb = in_dim // QK
    d = random_f16_normal_bits(g, n_tok * nb, -9, -4).reshape(n_tok, nb)
    q = g.integers(-127, 128, size=(n_tok, nb, QK))
    return make_blocks(d, q)


def pin_matmul_brute_force_exact(o):
    """Tiny shapes: fp32 result within the fp32-summation bound of the exact rational value."""
    g = rng(6)
    for in_dim, out_dim, n_tok in [(32, 1, 1), (64, 3, 2), (96, 3, 1), (160, 5, 3)]:
        W = _rand_weights(g, out_dim, in_dim)
        xq = _rand_acts(g, n_tok, in_dim)
        out, bound = o.matmul_q(W, xq, in_dim, out_dim, n_tok)
        ex, bd = exact_matmul(W, xq, in_dim, out_dim, n_tok)
        nb = in_dim // QK
        for t in range(n_tok):
            for r in range(out_dim):
                err = abs(Fraction(float(out[t, r])) - ex[t, r])
                lim = (nb + 2) * Fraction(1, 1 << 23) * bd[t, r]
                assert err <= lim, f"({in_dim},{out_dim},{n_tok}) t={t} o={r}: err {float(err)} > {float(lim)}"
                assert abs(bound[t, r] - float(bd[t, r])) <= 1e-12 * float(bd[t, r]) + 1e-300


def pin_matmul_double_dequant(o):
    """Against a float64 dequantise-then-dot (numpy matmul) within 1e-5 of the bound."""
    g = rng(7)
    in_dim, out_dim, n_tok = 256, 7, 4
    nb = in_dim // QK
    W = _rand_weights(g, out_dim, in_dim)
    xq = _rand_acts(g, n_tok, in_dim)
    dw, qw = split_blocks(W, nb)
    dx, qx = split_blocks(xq, nb)
    wf = (dw.view(np.float16).astype(np.float64)[..., None] * qw).reshape(out_dim, in_dim)
    xf = (dx.view(np.float16).astype(np.float64)[..., None] * qx).reshape(n_tok, in_dim)
    ref = xf @ wf.T
    out, bound = o.matmul_q(W, xq, in_dim, out_dim, n_tok)
    assert np.all(np.abs(out - ref) <= 1e-5 * bound + 1e-30)


def pin_matmul_integer_case(o):
    """Every scale 1.0: the result is the exact integer matrix product."""
    g = rng(8)
    in_dim, out_dim, n_tok = 128, 9, 5
    nb = in_dim // QK
    qw = g.integers(-127, 128, size=(out_dim, nb, QK))
    qx = g.integers(-127, 128, size=(n_tok, nb, QK))
    W = make_blocks(np.full((out_dim, nb), 0x3C00), qw)
    xq = make_blocks(np.full((n_tok, nb), 0x3C00), qx)
    out, _ = o.matmul_q(W, xq, in_dim, out_dim, n_tok)
    ref = qx.reshape(n_tok, in_dim).astype(np.int64) @ qw.reshape(out_dim, in_dim).astype(np.int64).T
    assert np.array_equal(out.astype(np.int64), ref)
    assert np.all(out == ref.astype(np.float32))


def pin_matmul_one_hot(o):
    """q_w = e_i, q_x = e_i in one block, zero elsewhere: out = d_w d_x exactly."""
    g = rng(9)
    in_dim, nb = 96, 3
    for trial in range(20):
        b = int(g.integers(0, nb))
        i = int(g.integers(0, QK))
        qw = np.zeros((1, nb, QK), dtype=np.int64)
        qx = np.zeros((1, nb, QK), dtype=np.int64)
        qw[0, b, i] = 1
        qx[0, b, i] = 1
        dw = random_f16_normal_bits(g, nb).reshape(1, nb)
        dx = random_f16_normal_bits(g, nb).reshape(1, nb)
        out, _ = o.matmul_q(make_blocks(dw, qw), make_blocks(dx, qx), in_dim, 1, 1)
        want = f16_exact(dw[0, b]) * f16_exact(dx[0, b])
        assert Fraction(float(out[0, 0])) == want


def pin_matmul_power_of_two_scaling(o):
    """Doubling every weight scale doubles every output exactly; a zero block adds exactly 0."""
    g = rng(10)
    in_dim, out_dim, n_tok = 192, 6, 3
    nb = in_dim // QK
    W = _rand_weights(g, out_dim, in_dim)
    xq = _rand_acts(g, n_tok, in_dim)
    out, _ = o.matmul_q(W, xq, in_dim, out_dim, n_tok)
    dw, qw = split_blocks(W, nb)
    W2 = make_blocks(dw + 0x0400, qw)  # exponent + 1
    out2, _ = o.matmul_q(W2, xq, in_dim, out_dim, n_tok)
    assert np.array_equal(out2, 2 * out)
    Wz = make_blocks(np.concatenate([dw, np.zeros((out_dim, 1), np.uint16)], 1),
                     np.concatenate([qw, np.zeros((out_dim, 1, QK), np.int8)], 1))
    dx, qx = split_blocks(xq, nb)
    xz = make_blocks(np.concatenate([dx, random_f16_normal_bits(g, n_tok).reshape(n_tok, 1)], 1),
                     np.concatenate([qx, g.integers(-127, 128, size=(n_tok, 1, QK)).astype(np.int8)], 1))
    outz, _ = o.matmul_q(Wz, xz, in_dim + QK, out_dim, n_tok)
    assert np.array_equal(outz, out)


def pin_matmul_orientation(o):
    """out[t][o] uses weight row o and activation row t (non-square, distinct rows)."""
    g = rng(11)
    in_dim, out_dim, n_tok = 64, 5, 2
    W = _rand_weights(g, out_dim, in_dim)
    xq = _rand_acts(g, n_tok, in_dim)
    out, _ = o.matmul_q(W, xq, in_dim, out_dim, n_tok)
    for t in range(n_tok):
        for r in range(out_dim):
            single, _ = o.matmul_q(W[r:r + 1], xq[t:t + 1], in_dim, 1, 1)
            assert single[0, 0] == out[t, r]
    ex, _ = exact_matmul(W, xq, in_dim, out_dim, n_tok)
    assert np.allclose(out, ex.astype(float), rtol=1e-5)


def pin_matmul_sample_consistent(o):
    """Sampled outputs equal the corresponding full-product outputs bit for bit."""
    g = rng(12)
    in_dim, out_dim, n_tok = 128, 11, 4
    W = _rand_weights(g, out_dim, in_dim)
    xq = _rand_acts(g, n_tok, in_dim)
    out, bound = o.matmul_q(W, xq, in_dim, out_dim, n_tok)
    tok = g.integers(0, n_tok, size=30)
    row = g.integers(0, out_dim, size=30)
    s, sb = o.matmul_sample(W, xq, in_dim, out_dim, n_tok, tok, row)
    assert np.array_equal(s, out[tok, row]) and np.array_equal(sb, bound[tok, row])
    ex, _ = exact_matmul(W, xq, in_dim, out_dim, n_tok)
    assert np.allclose(s, ex[tok, row].astype(float), rtol=1e-5)


def pin_quantize_then_matmul_brute(o):
    """End to end from fp32 x: quantise (checked by invariants) then the exact dot."""
    g = rng(13)
    in_dim, out_dim, n_tok = 64, 4, 3
    x = g.standard_normal((n_tok, in_dim)).astype(np.float32)
    W = _rand_weights(g, out_dim, in_dim)
    xq = o.quantize(x)
    out, bound = o.matmul(W, x, out_dim)
    ex, bd = exact_matmul(W, xq, in_dim, out_dim, n_tok)
    assert np.all(np.abs(out - ex.astype(float)) <= 1e-6 * bd.astype(float) + 1e-30)
    # the quantised dot approximates the unquantised fp64 dot within the quantisation error
    nb = in_dim // QK
    dw, qw = split_blocks(W, nb)
    wf = (dw.view(np.float16).astype(np.float64)[..., None] * qw).reshape(out_dim, in_dim)
    dxb, _ = split_blocks(xq, nb)
    step = dxb.view(np.float16).astype(np.float64)  # quantisation step per (t, b), error <= step/2 (+ fp16 rounding of d)
    lim = np.zeros((n_tok, out_dim))
    for b in range(nb):
        lim += (step[:, b:b + 1] * 0.5 * 1.01 + np.abs(x[:, b * QK:(b + 1) * QK]).max(1, keepdims=True) * 2 ** -10) \
            @ np.abs(wf[:, b * QK:(b + 1) * QK]).sum(1, keepdims=True).T
    assert np.all(np.abs(out - x.astype(np.float64) @ wf.T) <= lim)


# ---------------------------------------------------------------- routed experts
def pin_moe_identity_routing(o):
    """k = 1, token t -> expert t: each output row is that expert's matmul."""
    g = rng(14)
    n_exp, in_dim, out_dim = 4, 64, 6
    nb = in_dim // QK
    stride = out_dim * nb * QB + 16  # padded expert stride
    Wall = np.zeros(n_exp * stride, dtype=np.uint8)
    experts = []
    for e in range(n_exp):
        We = _rand_weights(g, out_dim, in_dim)
        experts.append(We)
        Wall[e * stride:e * stride + We.nbytes] = We.reshape(-1)
    xq = _rand_acts(g, n_exp, in_dim)
    ids = np.arange(n_exp, dtype=np.int32).reshape(n_exp, 1)
    out, bound, flag = o.moe(Wall, n_exp, stride, ids, in_dim, out_dim, xq, 0, n_exp)
    assert flag == 0
    for e in range(n_exp):
        ref, rb = o.matmul_q(experts[e], xq[e:e + 1], in_dim, out_dim, 1)
        assert np.array_equal(out[e], ref[0]) and np.array_equal(bound[e], rb[0])


def pin_moe_brute_force(o):
    """Random top-k routing, token rows and per-pair rows, against exact rationals."""
    g = rng(15)
    n_exp, in_dim, out_dim, n_tok, k = 5, 64, 3, 3, 2
    nb = in_dim // QK
    stride = out_dim * nb * QB
    Wall = _rand_weights(g, n_exp * out_dim, in_dim).reshape(-1)
    ids = np.stack([g.choice(n_exp, size=k, replace=False) for _ in range(n_tok)]).astype(np.int32)
    for per_pair in (0, 1):
        rows = n_tok * k if per_pair else n_tok
        xq = _rand_acts(g, rows, in_dim)
        out, bound, flag = o.moe(Wall, n_exp, stride, ids, in_dim, out_dim, xq, per_pair, n_tok)
        assert flag == 0
        for t in range(n_tok):
            for j in range(k):
                p = t * k + j
                e = int(ids[t, j])
                We = Wall[e * stride:(e + 1) * stride]
                xr = xq[p if per_pair else t]
                ex, bd = exact_matmul(We, xr, in_dim, out_dim, 1)
                err = np.array([abs(Fraction(float(out[p, r])) - ex[0, r]) for r in range(out_dim)])
                assert all(err[r] <= (nb + 2) * Fraction(1, 1 << 23) * bd[0, r] for r in range(out_dim)), (per_pair, t, j)
        pair = g.integers(0, n_tok * k, size=12)
        row = g.integers(0, out_dim, size=12)
        s, sb, sf = o.moe_sample(Wall, n_exp, stride, ids, in_dim, out_dim, xq, per_pair, n_tok, pair, row)
        assert sf == 0 and np.array_equal(s, out[pair, row])


def pin_moe_bad_ids(o):
    """Out-of-range expert ids give zero rows and raise the flag; valid pairs are unaffected."""
    g = rng(16)
    n_exp, in_dim, out_dim, n_tok, k = 3, 32, 4, 2, 2
    stride = out_dim * QB
    Wall = _rand_weights(g, n_exp * out_dim, in_dim).reshape(-1)
    xq = _rand_acts(g, n_tok, in_dim)
    ids = np.array([[0, 7], [-1, 2]], dtype=np.int32)
    out, _, flag = o.moe(Wall, n_exp, stride, ids, in_dim, out_dim, xq, 0, n_tok)
    assert flag == 1
    assert np.all(out[1] == 0) and np.all(out[2] == 0)
    ref0, _ = o.matmul_q(Wall[:stride], xq[0:1], in_dim, out_dim, 1)
    ref3, _ = o.matmul_q(Wall[2 * stride:3 * stride], xq[1:2], in_dim, out_dim, 1)
    assert np.array_equal(out[0], ref0[0]) and np.array_equal(out[3], ref3[0])


# ---------------------------------------------------------------- the expert FFN around the routed product
def _lambert_w(c: float) -> float:
    """Principal branch of Lambert's W at c > 0 (w e^w = c), by Newton's method."""
    w = 0.5
    for _ in range(60):
        ew = np.exp(w)
        w -= (w * ew - c) / (ew * (w + 1.0))
    return float(w)


def pin_swiglu_closed_forms(o):
    """silu at points with closed forms (no clamp): silu(0) = 0; at g = ln 3, e^-g = 1/3
    so silu(g) = (3/4) ln 3; silu(g) - silu(-g) = g; silu(g) = g to fp32 precision for
    large g and 0 for very negative g; the minimum of silu is -W(1/e), reached at
    g = -(1 + W(1/e)) (W: Lambert's function).  mid is linear in up."""
    u = np.array([1.0, -2.0, 0.5, 3.0], np.float32)
    assert np.all(o.swiglu(np.zeros(4, np.float32), u, 0.0) == 0)
    ln3 = np.float32(np.log(3.0))
    m = o.swiglu(np.full(4, ln3, np.float32), u, 0.0).astype(np.float64)
    ref = 0.75 * np.log(3.0) * u.astype(np.float64)
    assert np.all(np.abs(m - ref) <= 1e-6 * np.abs(ref))
    gs = np.linspace(-20.0, 20.0, 4001).astype(np.float32)
    ones = np.ones_like(gs)
    a = o.swiglu(gs, ones, 0.0).astype(np.float64)
    b = o.swiglu(-gs, ones, 0.0).astype(np.float64)
    assert np.all(np.abs(a - b - gs.astype(np.float64)) <= 2.0 ** -23 * (np.abs(a) + np.abs(b)) + 1e-30)
    big = np.array([40.0, 60.0, 88.0, 1000.0], np.float32)
    assert np.array_equal(o.swiglu(big, u, 0.0), big * u)
    neg = np.array([-120.0, -200.0, -1000.0, -1e30], np.float32)
    assert np.all(o.swiglu(neg, np.ones(4, np.float32), 0.0) == 0)
    w1e = _lambert_w(np.exp(-1.0))
    grid = np.linspace(-1.4, -1.15, 25001).astype(np.float32)
    mg = o.swiglu(grid, np.ones_like(grid), 0.0).astype(np.float64)
    assert abs(mg.min() + w1e) <= 1e-7
    assert abs(float(grid[np.argmin(mg)]) + 1.0 + w1e) <= 2e-3
    lin = o.swiglu(np.full(4, 1.5, np.float32), u, 0.0).astype(np.float64)
    assert np.all(np.abs(lin - lin[0] * u) <= 2.0 ** -22 * np.abs(lin))


def pin_swiglu_clamp(o):
    """The clamp (MoE page, SwiGLU activation section): gate is limited from above only,
    up to [-limit, limit]; values inside the band are unchanged; limit = 0 means none."""
    L = 10.0
    f = np.float32
    s = lambda g, u, lim: o.swiglu(np.array([g], f), np.array([u], f), lim)[0]
    for u in (1.0, -2.5, 7.0):
        assert s(50.0, u, L) == s(10.0, u, L)
        assert s(1e30, u, L) == s(10.0, u, L)
    for g in (-3.0, 0.7, 4.0):
        assert s(g, 50.0, L) == s(g, 10.0, L)
        assert s(g, -50.0, L) == s(g, -10.0, L)
        assert s(g, 9.5, L) == s(g, 9.5, 0.0)
        assert s(g, 50.0, L) != s(g, 50.0, 0.0)
    assert s(-50.0, 1.0, L) == s(-50.0, 1.0, 0.0)
    assert -1e-18 < s(-50.0, 1.0, L) < 0.0
    assert s(3.0, 2.0, L) == s(3.0, 2.0, 0.0)
    assert s(50.0, 1.0, 0.0) == 50.0
    assert abs(s(10.0, 1.0, L) - s(-10.0, 1.0, L) - 10.0) <= 2.0 ** -20


def pin_combine_integer_exact(o):
    """The weighted sum of a token's k expert rows, with integer rows and integer or
    dyadic weights: exact, equal to integer arithmetic; the bound is sum |w y|; k = 1
    with weight 1 returns the row."""
    g = rng(21)
    n_tok, k, dim = 3, 6, 40
    y = g.integers(-1000, 1001, size=(n_tok * k, dim))
    w = g.integers(-3, 4, size=n_tok * k)
    out, bound = o.combine(y.astype(np.float32), w.astype(np.float32), n_tok, k)
    yt, wt = y.reshape(n_tok, k, dim), w.reshape(n_tok, k)
    assert np.array_equal(out, np.einsum("tj,tjo->to", wt, yt).astype(np.float64))
    assert np.array_equal(bound, np.einsum("tj,tjo->to", np.abs(wt), np.abs(yt)).astype(np.float64))
    wd = g.choice([0.25, -0.5, 1.0, 2.0, -0.125], size=n_tok * k)
    out, _ = o.combine(y.astype(np.float32), wd.astype(np.float32), n_tok, k)
    ref = np.einsum("tj,tjo->to", (wd * 8).astype(np.int64).reshape(n_tok, k), yt) / 8.0
    assert np.array_equal(out, ref)
    out1, _ = o.combine(y[:4].astype(np.float32), np.ones(4, np.float32), 4, 1)
    assert np.array_equal(out1, y[:4].astype(np.float64))


def pin_moe_ffn_exact_construction(o):
    """A routed expert FFN whose every step is exact, against integer arithmetic.
    Token t's x is 127 at column c_t < 32 and 0 elsewhere, so it quantises to d = 1 and
    q = 127 e_{c_t}.  Every weight scale is 1 and block 0 of every gate row is all 1, so
    gate = 127 exactly, and silu(127) rounds to 127 (e^-127 is far below fp32
    resolution); up = 127 q_up[o][0][c_t] and mid = 16129 q_up[o][0][c_t].  The first
    row of every 32-row block of up holds +/-127 in block 0, so each 32-block of mid has
    scale 16129 exactly, quants q_up and stored binary16 scale 16128; then
    y = 16128 Q_down q_up, and out = sum_j w_j y_j with dyadic weights.  Swapping gate
    and up, feeding the down projection a token row, or mixing experts gives other
    values (q_up has negative entries; experts and tokens differ)."""
    g = rng(22)
    n_exp, in_dim, mid_dim, out_dim, n_tok, k = 5, 64, 96, 48, 4, 2
    nbi, nbm = in_dim // QK, mid_dim // QK
    one = 0x3C00
    qg = g.integers(-127, 128, size=(n_exp, mid_dim, nbi, QK))
    qg[:, :, 0, :] = 1
    qu = g.integers(-127, 128, size=(n_exp, mid_dim, nbi, QK))
    qu[:, ::QK, 0, :] = 127 * g.choice([-1, 1], size=(n_exp, mid_dim // QK, QK))
    qd = g.integers(-127, 128, size=(n_exp, out_dim, nbm, QK))
    blocks = lambda q, rows, nb: make_blocks(np.full((rows, nb), one, np.uint16), q.reshape(rows, nb, QK)).reshape(-1)
    Wg, Wu = blocks(qg, n_exp * mid_dim, nbi), blocks(qu, n_exp * mid_dim, nbi)
    Wd = blocks(qd, n_exp * out_dim, nbm)
    gu_stride, d_stride = mid_dim * nbi * QB, out_dim * nbm * QB
    ids = np.stack([g.choice(n_exp, size=k, replace=False) for _ in range(n_tok)]).astype(np.int32)
    w = g.choice([0.25, -0.5, 1.0, 2.0, 0.75], size=(n_tok, k)).astype(np.float32)
    c = g.integers(0, QK, size=n_tok)
    x = np.zeros((n_tok, in_dim), np.float32)
    x[np.arange(n_tok), c] = 127.0
    r = o.moe_ffn(Wg, Wu, Wd, n_exp, gu_stride, d_stride, ids, w, in_dim, mid_dim, out_dim, 0.0, x)
    assert r["flag"] == 0
    for t in range(n_tok):
        exact = np.zeros(out_dim, np.int64)
        tol = np.zeros(out_dim)
        for j in range(k):
            p, e = t * k + j, int(ids[t, j])
            qmid = qu[e, :, 0, c[t]]
            assert np.array_equal(r["mid"][p], (16129 * qmid).astype(np.float32)), (t, j)
            dm, qm = split_blocks(r["midq"][p], nbm)
            assert np.all(dm == 0x73E0) and np.array_equal(qm.reshape(-1), qmid)   # 16128 in binary16
            terms = 16128 * np.einsum("obi,bi->ob", qd[e], qmid.reshape(nbm, QK))
            yj = terms.sum(1)
            tol_j = (nbm + 1) * 2.0 ** -24 * np.abs(terms).sum(1)
            assert np.all(np.abs(r["y"][p].astype(np.float64) - yj) <= tol_j), (t, j)
            exact += (int(w[t, j] * 4) * yj)
            tol += abs(float(w[t, j])) * tol_j
        assert np.all(np.abs(r["out"][t] - exact / 4.0) <= tol), t


def pin_moe_ffn_bad_id(o):
    """A pair with an out-of-range expert id contributes nothing and raises the flag; the
    token's other pairs are unaffected."""
    g = rng(23)
    n_exp, in_dim, mid_dim, out_dim = 3, 64, 32, 8
    Wg = _rand_weights(g, n_exp * mid_dim, in_dim).reshape(-1)
    Wu = _rand_weights(g, n_exp * mid_dim, in_dim).reshape(-1)
    Wd = _rand_weights(g, n_exp * out_dim, mid_dim).reshape(-1)
    gu, ds = mid_dim * (in_dim // QK) * QB, out_dim * (mid_dim // QK) * QB
    x = g.standard_normal((1, in_dim)).astype(np.float32)
    w = np.array([[0.5, 0.25]], np.float32)
    good = o.moe_ffn(Wg, Wu, Wd, n_exp, gu, ds, np.array([[2, 1]], np.int32), w, in_dim, mid_dim, out_dim, 10.0, x)
    bad = o.moe_ffn(Wg, Wu, Wd, n_exp, gu, ds, np.array([[2, 9]], np.int32), w, in_dim, mid_dim, out_dim, 10.0, x)
    assert good["flag"] == 0 and bad["flag"] == 1
    assert np.all(bad["y"][1] == 0) and np.all(bad["mid"][1] == 0)
    assert np.array_equal(bad["y"][0], good["y"][0])
    assert np.array_equal(bad["out"][0], 0.5 * good["y"][0].astype(np.float64))


# ---------------------------------------------------------------- RMSNorm feeding the quantiser
def pin_rmsnorm_unit_rows(o):
    """Rows of +/-1 have mean square 1, so with a negligible eps y = x * gamma exactly (the
    scale 1/sqrt(1 + 2^-40) moves a value by far less than half an fp32 step); the
    quantised output is the quantiser of y."""
    g = rng(24)
    n_tok, dim = 3, 96
    x = g.choice([-1.0, 1.0], size=(n_tok, dim)).astype(np.float32)
    gamma = (0.5 + g.random(dim)).astype(np.float32)
    xq, y = o.rmsnorm_quantize(x, gamma, 2.0 ** -40)
    assert np.array_equal(y, x * gamma)
    assert np.array_equal(xq, o.quantize(y))
    xq1, y1 = o.rmsnorm_quantize(x, None, 2.0 ** -40)
    assert np.array_equal(y1, x)


def pin_rmsnorm_invariants(o):
    """Scale invariance under powers of two, the RMS of y / gamma equal to 1, the sign of
    x * gamma kept, linearity in gamma (power of two), and the limit where eps dominates."""
    g = rng(25)
    n_tok, dim = 4, 256
    x = g.standard_normal((n_tok, dim)).astype(np.float32)
    gamma = (1.0 + 0.2 * g.standard_normal(dim)).astype(np.float32)
    eps = 1e-30
    _, y = o.rmsnorm_quantize(x, gamma, eps)
    for k in (-3, 5):
        _, yk = o.rmsnorm_quantize(x * np.float32(2.0 ** k), gamma, eps)
        assert np.array_equal(yk, y)
    rms = np.sqrt(np.mean((y.astype(np.float64) / gamma) ** 2, axis=1))
    assert np.all(np.abs(rms - 1.0) <= 1e-6)
    assert np.all(np.sign(y) == np.sign(x * gamma))
    _, y2 = o.rmsnorm_quantize(x, 2 * gamma, eps)
    assert np.array_equal(y2, 2 * y)
    tiny = (1e-20 * x).astype(np.float32)            # mean square 1e-40, far below eps = 1
    _, yt = o.rmsnorm_quantize(tiny, gamma, 1.0)
    assert np.array_equal(yt, tiny * gamma)
    xq0, y0 = o.rmsnorm_quantize(np.zeros((2, dim), np.float32), gamma, 1e-6)
    assert np.all(y0 == 0) and np.all(xq0 == 0)


# ---------------------------------------------------------------- second weight format (K-quants x Q8_K)
QKK = 256
KQ_BYTES = {2: 84, 4: 144}


def _kq_golden():
    with open(os.path.join(GOLDEN, "kquant_worked.json")) as f:
        return json.load(f)


def _rand_kq(g, fmt, rows, in_dim):
    """Random K-quant rows: uniform bytes, then d and dmin set to binary16 normals of a few 2^-k."""
    nbk = in_dim // QKK
    raw = g.integers(0, 256, size=(rows, nbk, KQ_BYTES[fmt])).astype(np.uint8)
    off = 80 if fmt == 2 else 0
    for j in (0, 2):
        bits = random_f16_normal_bits(g, rows * nbk, -12, -6).reshape(rows, nbk)
        raw[..., off + j] = (bits & 0xFF).astype(np.uint8)
        raw[..., off + j + 1] = (bits >> 8).astype(np.uint8)
    return raw.reshape(rows, nbk * KQ_BYTES[fmt])


def pin_kq_dequant_golden(o):
    """Hand-derived weight values of hand-built Q2_K and Q4_K blocks (and one block sum)."""
    for b in _kq_golden()["kquant"]:
        w = o.kq_dequant(np.array(b["bytes"], np.uint8), b["fmt"], QKK, 1)[0]
        for k, v in b["values"].items():
            assert w[int(k)] == v, (b["name"], k, float(w[int(k)]), v)
        if "sum" in b:
            assert w.sum() == b["sum"], (b["name"], float(w.sum()))


def pin_kq_scale_doubling(o):
    """Doubling d and dmin (binary16 exponent + 1) doubles every weight; d = dmin = 0 zeroes them."""
    g = rng(42)
    for fmt in (2, 4):
        W = _rand_kq(g, fmt, 3, 512)
        W2 = W.copy().reshape(3, 2, KQ_BYTES[fmt])
        W0 = W2.copy()
        off = 80 if fmt == 2 else 0
        for j in (off, off + 2):
            bits = W2[..., j].astype(np.uint16) | (W2[..., j + 1].astype(np.uint16) << 8)
            bits = bits + (1 << 10)
            W2[..., j] = (bits & 0xFF).astype(np.uint8)
            W2[..., j + 1] = (bits >> 8).astype(np.uint8)
            W0[..., j] = 0
            W0[..., j + 1] = 0
        w = o.kq_dequant(W, fmt, 512, 3)
        assert np.array_equal(o.kq_dequant(W2.reshape(3, -1), fmt, 512, 3), 2 * w)
        assert not o.kq_dequant(W0.reshape(3, -1), fmt, 512, 3).any()


def pin_q8k_golden(o):
    """The Q8_K quantiser on hand-worked 256-value blocks."""
    for c in _kq_golden()["q8k"]:
        x = np.zeros((1, QKK), np.float32)
        x[0, :len(c["x_head"])] = c["x_head"]
        d, q = o.quantize_q8k(x)
        assert d[0, 0] == np.float32(c["d"]), (c["name"], float(d[0, 0]))
        n = len(c["q_head"])
        assert list(q[0, :n]) == c["q_head"] and not q[0, n:].any(), c["name"]


def pin_q8k_invariants(o):
    """|x/d - q| <= 1/2 in fp32, |q| <= 127 with 127 at the block maximum, sign symmetry,
    power-of-two scaling, zero blocks."""
    g = rng(43)
    x = (g.standard_normal((4, 1024)) * np.exp(g.uniform(-6, 6, size=(4, 1)))).astype(np.float32)
    x[1, 256:512] = 0.0
    d, q = o.quantize_q8k(x)
    for t in range(4):
        for b in range(4):
            blk = x[t, b * QKK:(b + 1) * QKK]
            qb = q[t, b * QKK:(b + 1) * QKK].astype(np.int64)
            if not blk.any():
                assert d[t, b] == 0 and not qb.any()
                continue
            assert np.abs(qb).max() == 127 and abs(qb[np.argmax(np.abs(blk))]) == 127
            quo = blk / np.float32(d[t, b])
            assert np.all(np.abs(quo.astype(np.float64) - qb) <= 0.5)
    dn, qn = o.quantize_q8k(-x)
    assert np.array_equal(dn, d) and np.array_equal(qn, -q)
    d4, q4 = o.quantize_q8k(x * np.float32(4))
    assert np.array_equal(d4, 4 * d) and np.array_equal(q4, q)


def pin_kq_matmul_exact(o):
    """Tiny shapes: the product is the fp32 rounding of the exact rational sum of dequantised
    weight times dequantised activation (weights from the golden-pinned dequantiser); the
    bound is at least the sum's magnitude."""
    g = rng(44)
    for fmt in (2, 4):
        for in_dim, out_dim, n_tok in [(256, 1, 1), (512, 3, 2), (768, 2, 3)]:
            W = _rand_kq(g, fmt, out_dim, in_dim)
            x = g.standard_normal((n_tok, in_dim)).astype(np.float32)
            dx, qx = o.quantize_q8k(x)
            out, bound = o.kq_matmul_q(W, fmt, in_dim, out_dim, dx, qx)
            w = o.kq_dequant(W, fmt, in_dim, out_dim)
            for t in range(n_tok):
                xs = [Fraction(float(dx[t, i // QKK])) * int(qx[t, i]) for i in range(in_dim)]
                for r in range(out_dim):
                    ex = sum(Fraction(float(w[r, i])) * xs[i] for i in range(in_dim))
                    slack = abs(ex) * Fraction(1, 1 << 23) + Fraction(float(bound[t, r])) * Fraction(1, 10 ** 12)
                    assert abs(Fraction(float(out[t, r])) - ex) <= slack, (fmt, in_dim, t, r)
                    assert bound[t, r] >= abs(float(ex)) * (1 - 1e-12)


def pin_kq_block_sum(o):
    """The hand-built Q2_K block against all-ones Q8_K activations (d_x = 1, q = 1): 3040."""
    b = [c for c in _kq_golden()["kquant"] if c["name"] == "q2k_fields"][0]
    W = np.array(b["bytes"] * 2, np.uint8).reshape(1, -1)
    out, _ = o.kq_matmul_q(W, 2, 512, 1, np.ones((1, 2), np.float32), np.ones((1, 512), np.int8))
    assert out[0, 0] == 2 * b["sum"]


def pin_kq_moe_brute(o):
    """Routed K-quant experts: each pair equals the dense product of its expert and its row;
    bad ids give zero rows and raise the flag."""
    g = rng(45)
    for fmt in (2, 4):
        n_exp, in_dim, out_dim, n_tok, k = 4, 512, 3, 3, 2
        stride = out_dim * in_dim // QKK * KQ_BYTES[fmt]
        Wall = _rand_kq(g, fmt, n_exp * out_dim, in_dim).reshape(-1)
        ids = np.array([[0, 3], [2, 1], [3, 9]], dtype=np.int32)
        for per_pair in (0, 1):
            x = g.standard_normal((n_tok * k if per_pair else n_tok, in_dim)).astype(np.float32)
            out, bound, flag = o.kq_moe(Wall, fmt, n_exp, stride, ids, in_dim, out_dim, x, per_pair)
            assert flag == 1 and not out[5].any()
            for p in range(5):
                e = int(ids.reshape(-1)[p])
                xr = x[p if per_pair else p // k][None]
                ref, _ = o.kq_matmul(Wall[e * stride:(e + 1) * stride], fmt, xr, out_dim)
                assert np.array_equal(out[p], ref[0]), (fmt, per_pair, p)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
