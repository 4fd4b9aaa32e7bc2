"""Pins of the oracle's logarithmic and differential quantisation
('分布式训练中的梯度压缩算法' 二.1 对数量化 and 二.4 差分量化).

Log quantisation: the binary32 log and exp (Cody-Waite) against the true
functions, a hand-worked case, and agreement with the page's formula
restated here in float64 numpy away from rounding ties.  Differential
quantisation: a hand case, refresh = plain EF quantisation, the receiver's
history equal to the sender's, the per-step error bound of the closed loop
and the error-feedback identity."""
import math

import numpy as np
import pytest

import oracle

f32 = np.float32


def ulps(got, true):
    return abs(float(got) - true) / float(np.spacing(f32(abs(true))))


def test_log_exp_accuracy():
    r = np.random.default_rng(0)
    xs = np.concatenate([1 + r.random(3000) * 0.01, 1 + r.random(3000), 1 + r.random(3000) * 1e3,
                         np.exp(r.random(3000) * 85)]).astype(f32)
    worst = max(ulps(oracle.logf(x), math.log(float(x))) for x in xs if x > 1)
    assert worst <= 2.0, worst
    ys = np.concatenate([r.random(3000), r.random(3000) * 88.0, np.arange(0, 88, 0.05)]).astype(f32)
    worst = max(ulps(oracle.expf(y), math.exp(float(y))) for y in ys)
    assert worst <= 1.5, worst


def test_log_exp_exact_points():
    assert oracle.logf(1.0) == 0.0
    assert oracle.expf(0.0) == 1.0
    for k in range(1, 60, 7):
        assert ulps(oracle.logf(2.0 ** k), k * math.log(2.0)) <= 1.0
        y = f32(k * math.log(2.0))
        assert ulps(oracle.expf(y), math.exp(float(y))) <= 1.5


def test_log_hand_case():
    # 4 bits: sign + 3 magnitude bits, 7 levels; max |x| = 3 so scale =
    # log(4) / 7 and log(|x| + 1) / scale = 7, 3.98, 0, 1.70 -> 7, 4, 0, 2
    x = np.array([3.0, -1.2, 0.0, 0.4], f32)
    codes, scales = oracle.quant(x, 4, 0, "log")
    assert codes[:2].tolist() == [7 | (12 << 4), 0 | (2 << 4)]  # sign-magnitude nibbles
    assert abs(float(scales[0]) - math.log(4.0) / 7) <= 2e-7
    g_hat = oracle.dequant(codes, scales, 4, 4, 0, "log")
    s = math.log(4.0) / 7
    want = [math.exp(7 * s) - 1, -(math.exp(4 * s) - 1), 0.0, math.exp(2 * s) - 1]
    for g, w in zip(g_hat, want):
        assert abs(float(g) - w) <= 8 * float(np.spacing(f32(max(abs(w), 1.0))))
    assert not np.signbit(g_hat[2])


@pytest.mark.parametrize("bits,group", [(8, 0), (4, 64), (2, 16)])
def test_log_matches_the_page_formula(bits, group):
    """q = sign(g) round(log(|g| + 1) / scale), scale = log(max|g| + 1) /
    (2^(b-1) - 1), g_hat = sign(q) (exp(|q| scale) - 1), evaluated in float64
    from the formula: the codes agree wherever t is not within 1e-3 of a
    rounding tie, g_hat within 1e-5 relative."""
    r = np.random.default_rng(bits)
    n = 4096
    x = (r.standard_normal(n) * 10).astype(f32)
    codes, scales = oracle.quant(x, bits, group, "log")
    g_hat = oracle.dequant(codes, scales, n, bits, group, "log")
    G = n if group == 0 else group
    lv = 2 ** (bits - 1) - 1
    xd = x.astype(np.float64).reshape(-1, G)
    scale = np.log(np.abs(xd).max(axis=1, keepdims=True) + 1) / lv
    t = np.log(np.abs(xd) + 1) / scale
    q = np.sign(xd) * np.round(t)
    far = (np.abs(t - np.floor(t) - 0.5) > 1e-3).reshape(-1)
    mask = (1 << (bits - 1)) - 1
    raw = np.unpackbits(codes[:n * bits // 8], bitorder="little").reshape(-1, bits)
    code = (raw * (1 << np.arange(bits))).sum(axis=1)
    got_q = np.where(code >> (bits - 1), -1, 1) * (code & mask)
    assert np.array_equal(got_q[far], q.reshape(-1)[far].astype(int))
    want = (np.sign(q) * (np.exp(np.abs(q) * scale) - 1)).reshape(-1)
    assert np.allclose(g_hat[far], want[far], rtol=1e-5, atol=1e-30)


def test_log_rejects_one_bit():
    with pytest.raises(oracle.OracleError):
        oracle.quant(np.ones(8, f32), 1, 0, "log")


def test_diff_hand_case():
    g = np.array([1, 2, 3, 4], f32)
    ref = np.ones(4, f32)
    codes, scales, e2, ref2 = oracle.ef_diff_quant(g, np.zeros(4, f32), ref, 2, 0, "minmax")
    assert scales.tolist() == [1.0, 0.0]          # d = [0, 1, 2, 3]: scale 1, min 0
    assert codes[0] == 0 | (1 << 2) | (2 << 4) | (3 << 6)
    assert ref2.tolist() == g.tolist() and not np.any(e2)


@pytest.mark.parametrize("mode,bits", [("minmax", 4), ("qsgd", 8), ("log", 8)])
def test_refresh_is_plain_quantisation(mode, bits):
    r = np.random.default_rng(1)
    g = r.standard_normal(1000).astype(f32)
    e = (0.1 * r.standard_normal(1000)).astype(f32)
    ref = r.standard_normal(1000).astype(f32)
    c1, s1, e1, ref1 = oracle.ef_diff_quant(g, e, ref, bits, 64, mode, "stochastic", 3, 2,
                                            refresh=True)
    c2, s2, e2 = oracle.ef_quant(g, e, bits, 64, mode, "stochastic", 3, 2)
    assert np.array_equal(c1, c2) and np.array_equal(s1.view(np.uint32), s2.view(np.uint32))
    assert np.array_equal(e1.view(np.uint32), e2.view(np.uint32))
    g_hat = (f32(0) + oracle.dequant(c1, s1, 1000, bits, 64, mode)).astype(f32)
    assert np.array_equal(ref1.view(np.uint32), g_hat.view(np.uint32))


@pytest.mark.parametrize("mode,bits", [("minmax", 4), ("qsgd", 4), ("log", 4)])
def test_closed_loop_over_steps(mode, bits):
    """Correlated steps without error feedback: the receiver's history equals
    the sender's bit for bit, and each step's reconstruction error is the
    quantisation error of that step's difference only (no pile-up)."""
    n, G = 2048, 64
    r = np.random.default_rng(2)
    g = r.standard_normal(n).astype(f32)
    ref_s = np.zeros(n, f32)
    ref_r = np.zeros(n, f32)
    for step in range(12):
        g = (0.9 * g + 0.3 * r.standard_normal(n)).astype(f32)
        refresh = step % 5 == 0
        r_old = np.zeros(n, f32) if refresh else ref_s.copy()
        d = (g - r_old).astype(f32)
        codes, scales, _, ref_s = oracle.ef_diff_quant(g, None, ref_s, bits, G, mode,
                                                       "nearest_even", 0, step, refresh)
        ref_r = oracle.diff_dequant(codes, scales, ref_r, n, bits, G, mode, refresh)
        assert np.array_equal(ref_s.view(np.uint32), ref_r.view(np.uint32))
        d_hat = oracle.dequant(codes, scales, n, bits, G, mode)
        # g - ref' = (d - d_hat) + the roundings of d = g - r and ref' = r + d_hat
        err = np.abs(g.astype(np.float64) - ref_s)
        qerr = np.abs(d.astype(np.float64) - d_hat)
        big = np.maximum.reduce([np.abs(g), np.abs(r_old), np.abs(ref_s), np.abs(d)])
        slack = np.spacing(big).astype(np.float64)
        assert np.all(err <= qerr + slack)


def test_error_feedback_identity():
    r = np.random.default_rng(3)
    g = r.standard_normal(3000).astype(f32)
    e = (0.2 * r.standard_normal(3000)).astype(f32)
    ref = r.standard_normal(3000).astype(f32)
    _, _, e2, ref2 = oracle.ef_diff_quant(g, e.copy(), ref, 2, 32, "qsgd", "stochastic", 9, 1)
    c = (g + e).astype(f32)
    assert np.array_equal(e2.view(np.uint32), (c - ref2).astype(f32).view(np.uint32))
