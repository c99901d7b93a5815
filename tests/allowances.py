"""Agreement rules for RMSNorm feeding the quantiser, shared by its GPU parity test
and the CPU test of the rules themselves (tests/test_tolerances.py).

The kernel's sum of squares has relative error at most n_s 2^-24 with
n_s = 8 ceil(dim/2048) + 14 (its fixed reduction order); the mean, + eps, sqrt,
reciprocal, two products and the oracle's own rounding add at most 7 roundings,
and sqrt halves the sum's error: ((n_s + 2) / 2 + 5) 2^-24 to first order, and
rho adds one more 2^-24 for the second-order terms.  From there:

* y: |y_gpu - y_oracle| <= rho |y_oracle| + 1e-37;
* quants: equal, or 1 apart where the oracle's |y/d| lies within
  max(1e-3, 3 (2 rho + 2^-22) 127) of a rounding tie (three times the largest
  movement of y/d);
* binary16 scales: equal, or one step apart where the oracle's fp32
  d = amax/127 lies within 4 rho of a binary16 rounding midpoint.
"""
import math

import numpy as np

QK, QB = 32, 34


def rms_rho(dim: int) -> float:
    n_s = 8 * math.ceil(dim / 2048) + 14
    return ((n_s + 2) / 2 + 6) * 2.0 ** -24


def split_blocks(xq, nb):
    r = np.asarray(xq).reshape(-1, nb, QB)
    d = r[..., 0].astype(np.uint16) | (r[..., 1].astype(np.uint16) << 8)
    q = r[..., 2:].copy().view(np.int8).astype(np.int32)
    return d, q


def f16_near_midpoint(d32, rel):
    """True where the fp32 value lies within rel (relative) of a binary16 rounding midpoint."""
    d = d32.astype(np.float64)
    h16 = d32.astype(np.float16)
    h = h16.astype(np.float64)
    up = np.nextafter(h16, np.float16(np.inf)).astype(np.float64)
    dn = np.nextafter(h16, np.float16(0)).astype(np.float64)
    mids = np.stack([(h + up) / 2, (h + dn) / 2])
    return np.any(np.abs(mids - d) <= rel * np.abs(d), axis=0)


def check_rmsnorm(xq, y, xq_o, y_o):
    """Raise AssertionError unless (xq, y) from the kernel agree with the oracle's (xq_o, y_o)
    under the rules above.  xq: uint8 [n_tok, dim/32*34]; y: float [n_tok, dim]."""
    y = np.asarray(y, dtype=np.float64)
    n_tok, dim = y.shape
    nb = dim // QK
    r = rms_rho(dim)
    err = np.abs(y - y_o)
    assert np.all(err <= r * np.abs(y_o) + 1e-37), f"y: worst relative {np.max(err / (np.abs(y_o) + 1e-30)):.3e}"
    dg, qg = split_blocks(xq, nb)
    do, qo = split_blocks(xq_o, nb)
    d32 = np.abs(np.asarray(y_o, np.float32).reshape(n_tok, nb, QK)).max(-1) / np.float32(127.0)
    near_mid = f16_near_midpoint(d32, 4 * r)
    dgf = dg.view(np.float16).astype(np.float64)
    dof = do.view(np.float16).astype(np.float64)
    step = np.abs(np.nextafter(do.view(np.float16), np.float16(np.inf)).astype(np.float64) - dof)
    assert np.all((dg == do) | (near_mid & (np.abs(dgf - dof) <= step))), "binary16 scale differs away from a midpoint"
    window = max(1e-3, 3 * (2 * r + 2.0 ** -22) * 127)
    with np.errstate(divide="ignore", invalid="ignore"):
        quo = np.abs(np.asarray(y_o, np.float64).reshape(n_tok, nb, QK) / d32[..., None].astype(np.float64))
    near_tie = np.abs(quo - np.floor(quo) - 0.5) < window
    diff = qg != qo
    assert np.all(np.abs(qg - qo) <= 1), "a quant differs by more than 1"
    assert np.all(~diff | near_tie), f"{np.sum(diff & ~near_tie)} quants differ away from a tie"
