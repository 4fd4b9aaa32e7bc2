"""Pins of the oracle's diagnostics ('gradient-compression-quantization-
sparsification' 3.2: the gradient norm ratio after / before compression;
'梯度聚合通信优化实战方案' Python 演示: the error energy sum(err**2)): a
hand-worked case, exact rational sums on random buckets, the Top-K energy
split, the limits k = 0 and k = n, and agreement with the residual the
compressor itself stores."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _exact(vals):
    """Exact sum of squares of binary32 values as a Fraction."""
    return sum((Fraction(float(v)) ** 2 for v in vals), Fraction(0))


def _close(got, exact, n):
    """binary64 running sum of n exact binary64 squares: relative error at
    most (n - 1) * 2^-53 (n = 0: exactly zero)."""
    tol = float(exact) * (max(n, 1) * 2.0 ** -53) + 1e-300
    assert abs(Fraction(float(got)) - exact) <= Fraction(tol), (got, float(exact))


def test_hand_case():
    # g = [0.5, -2, 1, -1, 0.25, 2], k = 3: kept [1, 2, 5] = [-2, 1, 2]
    g = np.array([0.5, -2, 1, -1, 0.25, 2], np.float32)
    idx, val, _ = oracle.ef_topk(g, np.zeros_like(g), 3)
    d = oracle.diagnostics(g, np.zeros_like(g), idx, val)
    assert d.tolist() == [10.3125, 9.0, 1.3125]
    assert math.isclose(math.sqrt(d[1] / d[0]), math.sqrt(9 / 10.3125))


@pytest.mark.parametrize("n,k", [(1009, 10), (4096, 4096), (3000, 0), (777, 1)])
def test_topk_exact_sums(n, k):
    r = np.random.default_rng(n + k)
    g = r.standard_normal(n).astype(np.float32)
    e = (0.3 * r.standard_normal(n)).astype(np.float32)
    c = g + e  # binary32, as the compressor adds
    idx, val, err2 = oracle.ef_topk(g, e.copy(), k)
    d = oracle.diagnostics(g, e, idx, val)
    _close(d[0], _exact(c), n)
    _close(d[1], _exact(val), k)
    _close(d[2], _exact(err2), n)
    # Top-K moves energy, it does not change it: sum c^2 = kept + residual
    assert _exact(c) == _exact(val) + _exact(err2)
    if k == 0:
        assert d[1] == 0.0 and d[2] == d[0]
    if k == n:
        assert d[2] == 0.0 and d[1] == d[0]


@pytest.mark.parametrize("bits,group", [(8, 64), (2, 4)])
def test_hybrid_matches_the_stored_residual(bits, group):
    """For the hybrid, g_hat is the dequantised kept values and e' the
    residual ef_topk_quant stores."""
    n, k = 5000, 300
    r = np.random.default_rng(bits)
    g = r.standard_normal(n).astype(np.float32)
    e = (0.2 * r.standard_normal(n)).astype(np.float32)
    idx, codes, scales, err2 = oracle.ef_topk_quant(g, e.copy(), k, bits, group,
                                                    "stochastic", 7, 1)
    g_hat = oracle.dequant(codes, scales, k, bits, group, "qsgd")
    d = oracle.diagnostics(g, e, idx, g_hat)
    _close(d[0], _exact(g + e), n)
    _close(d[1], _exact(g_hat), k)
    _close(d[2], _exact(err2), n)
    assert d[1] < d[0]


def test_without_residual_is_the_error_of_the_transmitted_values():
    g = np.array([3.0, -1.0, 0.5, 4.0], np.float32)
    d = oracle.diagnostics(g, None, np.array([0, 3], np.int32), np.array([2.5, 4.0], np.float32))
    assert d.tolist() == [9 + 1 + 0.25 + 16, 6.25 + 16, 0.25 + 1 + 0.25 + 0]


def test_rejects_bad_indices():
    g = np.ones(5, np.float32)
    for bad in ([3, 1], [0, 5], [2, 2]):
        with pytest.raises(oracle.OracleError):
            oracle.diagnostics(g, None, np.array(bad, np.int32), np.ones(2, np.float32))
