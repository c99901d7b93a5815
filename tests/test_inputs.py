"""The seeded input generator: determinism and the stated distributions (no GPU)."""
import numpy as np

import inputs


def test_weights_deterministic_and_in_range():
    a = inputs.weights(64, 256, seed=0)
    b = inputs.weights(64, 256, seed=0)
    c = inputs.weights(64, 256, seed=1)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    blk = a.reshape(-1, 34)
    d = (blk[:, 0].astype(np.uint16) | (blk[:, 1].astype(np.uint16) << 8)).view(np.float16).astype(np.float64)
    assert d.min() >= 1e-3 - 1e-6 and d.max() <= 1e-2 + 1e-5
    q = blk[:, 2:].view(np.int8).astype(np.int64)
    assert q.min() == -127 and q.max() == 127
    assert abs(q.mean()) < 1.0 and abs(q.std() - np.sqrt((255 ** 2 - 1) / 12)) < 1.0


def test_weights_slices_are_independent_of_total():
    """Counter-based: the first rows do not depend on how many rows are drawn."""
    a = inputs.weights(8, 128, seed=3)
    b = inputs.weights(40, 128, seed=3)
    assert np.array_equal(a, b[:8])


def test_normal_moments_and_outliers():
    x = inputs.normal((400, 1000), seed=0)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    y = inputs.normal((400, 1000), seed=0, p_out=0.01, out_scale=20.0)
    ratio = y / x
    frac = np.mean(np.isclose(ratio, 20.0))
    assert 0.008 < frac < 0.012
    assert np.all(np.isclose(ratio, 1.0) | np.isclose(ratio, 20.0))


def test_routing_uniform_distinct():
    ids = inputs.route_uniform(64, 6, 256, seed=0)
    assert ids.shape == (64, 6) and ids.min() >= 0 and ids.max() < 256
    assert all(len(set(r)) == 6 for r in ids.tolist())
    assert 150 < len(np.unique(ids)) < 250


def test_routing_zipf_skew():
    ids = inputs.route_zipf(4096, 6, 256, s=1.1, seed=0)
    assert all(len(set(r)) == 6 for r in ids[:200].tolist())
    counts = np.bincount(ids.reshape(-1), minlength=256)
    assert counts[0] == 4096 or counts[0] > 3000  # the top-ranked expert is nearly always chosen
    assert counts[0] >= counts[10] >= counts[100] and counts.sum() == 4096 * 6
    assert (counts > 0).sum() == 256


def test_kquant_weights_deterministic_and_in_range():
    """K-quant rows: d and dmin on the binary16 grid inside the stated ranges, other bytes uniform,
    counter-based (a prefix does not depend on the total)."""
    for fmt, bb, off in ((2, 84, 80), (4, 144, 0)):
        a = inputs.kq_weights(32, 512, fmt, seed=0)
        assert a.shape == (32, 2 * bb)
        assert np.array_equal(a, inputs.kq_weights(32, 512, fmt, seed=0))
        assert not np.array_equal(a, inputs.kq_weights(32, 512, fmt, seed=1))
        assert np.array_equal(inputs.kq_weights(4, 512, fmt, seed=0), a[:4])
        blk = a.reshape(-1, bb)
        d_lo, d_hi, m_lo, m_hi = inputs.KQ_SCALES[fmt]
        for j, (lo, hi) in ((off, (d_lo, d_hi)), (off + 2, (m_lo, m_hi))):
            v = (blk[:, j].astype(np.uint16) | (blk[:, j + 1].astype(np.uint16) << 8)).view(np.float16)
            v = v.astype(np.float64)
            assert v.min() >= lo * (1 - 1e-3) and v.max() <= hi * (1 + 1e-3)
        rest = np.delete(blk, [off, off + 1, off + 2, off + 3], axis=1).astype(np.float64)
        assert abs(rest.mean() - 127.5) < 3.0 and rest.min() == 0 and rest.max() == 255
