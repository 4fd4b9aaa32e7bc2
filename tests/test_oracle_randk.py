"""Pins of the oracle's random sparsification with error feedback
('分布式训练中的梯度压缩算法' 二.2 随机稀疏化: keep an element with
probability p): the keep set recomputed from the Philox draw (itself pinned
by the published known-answer vectors), the limits p = 0 and p = 1, the
binomial statistics of the page's mask, and the residual bookkeeping."""
import numpy as np
import pytest

import oracle


def _c(g, e):
    return (g + e).astype(np.float32) if e is not None else g


@pytest.mark.parametrize("n,p,seed,step", [(1000, 0.1, 3, 0), (4097, 0.01, 7, 5),
                                           (333, 0.5, 11, 2), (1, 0.9, 0, 0)])
def test_keep_set_is_the_philox_draw_below_p(n, p, seed, step):
    r = np.random.default_rng(n)
    g = r.standard_normal(n).astype(np.float32)
    e = (0.1 * r.standard_normal(n)).astype(np.float32)
    c = _c(g, e)
    idx, val, e2 = oracle.ef_randk(g, e.copy(), p, seed, step)
    want = [i for i in range(n) if oracle.uniform(seed, step, i) < np.float32(p)]
    assert idx.tolist() == want
    assert np.array_equal(val.view(np.uint32), c[want].view(np.uint32))
    ref = c.copy()
    ref[want] = 0.0
    assert np.array_equal(e2.view(np.uint32), ref.view(np.uint32))  # kept are +0


def test_limits():
    g = np.linspace(-1, 1, 257).astype(np.float32)
    idx, val, e2 = oracle.ef_randk(g, np.zeros_like(g), 0.0, 1, 1)
    assert idx.size == 0 and np.array_equal(e2, g)
    idx, val, e2 = oracle.ef_randk(g, np.zeros_like(g), 1.0, 1, 1)
    assert idx.tolist() == list(range(g.size)) and np.array_equal(val, g)
    assert not np.any(e2) and not np.any(np.signbit(e2))


def test_fraction_matches_the_pages_mask_statistics():
    """The page's mask rand(n) < p keeps Binomial(n, p) entries: the count
    lies within 5 standard deviations, and two steps are independent."""
    n, p = 200_000, 0.01
    g = np.ones(n, np.float32)
    i0, _, _ = oracle.ef_randk(g, None, p, 42, 0)
    i1, _, _ = oracle.ef_randk(g, None, p, 42, 1)
    sd = np.sqrt(n * p * (1 - p))
    assert abs(i0.size - n * p) < 5 * sd
    both = np.intersect1d(i0, i1).size
    assert abs(both - n * p * p) < 5 * np.sqrt(n * p * p) + 2


def test_without_residual():
    g = np.arange(50, dtype=np.float32)
    idx, val, e2 = oracle.ef_randk(g, None, 0.3, 9, 9)
    assert e2 is None and np.array_equal(val, g[idx])
