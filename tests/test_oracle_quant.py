"""Pins of the oracle's quantise / dequantise / EF-quantise against hand-worked
cases, error bounds, unbiasedness, exact packing checked by numpy's bit
routines, the pages' own NumPy listing of linear quantisation, and the
error-feedback identity."""
import json
import os

import numpy as np
import pytest

import oracle

U = 2.0 ** -24  # unit roundoff of binary32


def _hex(v):
    return np.array([float.fromhex(x) for x in v], np.float32)


def _golden(golden_dir):
    return json.load(open(os.path.join(golden_dir, "quant_hand.json")))["cases"]


def test_hand_cases(golden_dir):
    for case in _golden(golden_dir):
        x = _hex(case["x"])
        bits, group, mode = case["bits"], case["group"], case["mode"]
        codes, scales = oracle.quant(x, bits, group, mode)
        assert np.array_equal(scales.view(np.uint32),
                              _hex(case["scales"]).view(np.uint32)), case["name"]
        want = case["codes"]
        assert codes[:len(want)].tolist() == want, case["name"]
        mag = (x.size * bits + 7) // 8
        assert not codes[len(want):mag].any(), case["name"]
        if "signs" in case:
            sign_off = (mag + 15) // 16 * 16
            assert codes[sign_off:sign_off + len(case["signs"])].tolist() == \
                case["signs"], case["name"]
        if "x_hat" in case:
            xh = oracle.dequant(codes, scales, x.size, bits, group, mode)
            assert np.array_equal(xh.view(np.uint32),
                                  _hex(case["x_hat"]).view(np.uint32)), case["name"]
        if "err" in case:
            c2, s2, e2 = oracle.ef_quant(x, np.zeros_like(x), bits, group, mode)
            assert np.array_equal(c2, codes) and np.array_equal(s2, scales)
            assert np.array_equal(e2, _hex(case["err"])), case["name"]


def test_sizes():
    # 8-bit codes are 1/4 and 4-bit codes 1/8 of fp32 (4、梯度累积与梯度压缩
    # 4.2.2); INT8 is 4x and 1-bit 32x (梯度聚合通信优化实战方案 梯度压缩原理).
    n = 1 << 20
    for bits in (1, 2, 4, 8):
        assert 32 * n / (8 * oracle.codes_bytes(n, bits, "minmax")) == 32 / bits
        assert 32 * n / (8 * oracle.codes_bytes(n, bits, "qsgd")) == 32 / (bits + 1)
    assert 32 * n / (8 * oracle.codes_bytes(n, 2, "tern")) == 16
    assert oracle.codes_bytes(5, 8, "minmax") == 16
    assert oracle.codes_bytes(17, 8, "qsgd") == 32 + 16
    assert oracle.scales_floats(130, 64, "minmax") == 6
    assert oracle.scales_floats(130, 64, "qsgd") == 3
    assert oracle.scales_floats(130, 0, "tern") == 1
    assert oracle.scales_floats(0, 64, "qsgd") == 0


@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_packing_is_little_endian_bitstream(bits):
    """Integer inputs spanning [0, 2^b - 1] have scale 1 and codes equal to
    the inputs, so numpy's unpackbits must give them back."""
    r = np.random.default_rng(bits)
    n = 1003
    top = (1 << bits) - 1
    q = r.integers(0, top + 1, size=n)
    q[0], q[1] = 0, top
    codes, scales = oracle.quant(q.astype(np.float32), bits, 0, "minmax")
    assert scales.tolist() == [1.0, 0.0]
    bitstream = np.unpackbits(codes, bitorder="little")[:n * bits]
    fields = bitstream.reshape(n, bits)
    got = (fields * (1 << np.arange(bits))).sum(axis=1)
    assert np.array_equal(got, q)
    assert not np.unpackbits(codes, bitorder="little")[n * bits:].any()


def test_qsgd_sign_plane():
    r = np.random.default_rng(5)
    x = r.standard_normal(777).astype(np.float32)
    codes, scales = oracle.quant(x, 4, 64, "qsgd")
    mag = (777 * 4 + 7) // 8
    signs = np.unpackbits(codes[(mag + 15) // 16 * 16:], bitorder="little")[:777]
    q = np.unpackbits(codes[:mag], bitorder="little")[:777 * 4].reshape(777, 4)
    q = (q * (1 << np.arange(4))).sum(axis=1)
    assert np.array_equal(signs.astype(bool), (x < 0) & (q != 0))


@pytest.mark.parametrize("G", [64, 1000, 0])
@pytest.mark.parametrize("bits", [1, 4, 8])
def test_nearest_error_bound(G, bits):
    """|g_hat - x| <= scale / 2 (plus rounding slack) for nearest rounding."""
    r = np.random.default_rng(G + bits)
    x = (r.standard_normal(5000) * 0.01).astype(np.float32)
    x[r.integers(0, 5000, 5)] *= 100
    codes, scales = oracle.quant(x, bits, G, "minmax")
    xh = oracle.dequant(codes, scales, x.size, bits, G, "minmax")
    g = G or x.size
    sc = np.repeat(scales[0::2], g)[:x.size].astype(np.float64)
    mn = np.repeat(scales[1::2], g)[:x.size].astype(np.float64)
    slack = 8 * U * (np.abs(x) + np.abs(mn) + sc * (2 ** bits))
    assert np.all(np.abs(xh.astype(np.float64) - x) <= 0.5 * sc + slack)
    # QSGD: |g_hat - x| <= scale / 2 on the magnitude
    codes, scales = oracle.quant(x, bits, G, "qsgd")
    xh = oracle.dequant(codes, scales, x.size, bits, G, "qsgd")
    sc = np.repeat(scales, g)[:x.size].astype(np.float64)
    slack = 8 * U * (np.abs(x) + sc * (2 ** bits))
    assert np.all(np.abs(xh.astype(np.float64) - x) <= 0.5 * sc + slack)


def test_qsgd_norm_within_tree_bound():
    """The group norm is within the summation error bound of the exact norm
    (a dropped or doubled term would be far outside it)."""
    r = np.random.default_rng(11)
    for G in (64, 100, 4096):
        x = r.standard_normal(G * 3 + 17).astype(np.float32)
        _, scales = oracle.quant(x, 8, G, "qsgd")
        for g in range(scales.size):
            xs = x[g * G:(g + 1) * G].astype(np.float64)
            exact = np.sqrt(np.sum(xs * xs))
            depth = int(np.ceil(np.log2(max(xs.size, 2)))) + 2
            assert abs(scales[g] * 255.0 - exact) <= (depth + 2) * U * exact + \
                255.0 * U * scales[g]


def test_matches_pages_numpy_listing():
    """For 8-bit nearest min-max on one group the oracle agrees bit for bit
    with the linear_quantize listing of 分布式训练中的梯度压缩算法 二.1
    evaluated in numpy float32 (np.round is half to even)."""
    r = np.random.default_rng(2)
    for n in (10, 1000, 65536):
        x = r.standard_normal(n).astype(np.float32)
        mn, mx = x.min(), x.max()
        scale = (mx - mn) / np.float32(2 ** 8 - 1)
        q = np.round((x - mn) / scale)
        g_hat = q * scale + mn
        codes, scales = oracle.quant(x, 8, 0, "minmax")
        xh = oracle.dequant(codes, scales, n, 8, 0, "minmax")
        assert scales[0] == scale and scales[1] == mn
        assert np.array_equal(codes[:n], q.astype(np.uint8))
        assert np.array_equal(xh, g_hat.astype(np.float32))
        # the demo's .astype(np.int8) wraps codes above 127; unsigned codes
        # keep them (reading of 梯度聚合通信优化实战方案 Python 演示)
        assert codes[:n].max() == 255


@pytest.mark.parametrize("mode", ["minmax", "qsgd", "tern"])
def test_stochastic_unbiased(mode):
    """Mean of g_hat over many (seed) draws converges to x
    (hotdry 'gradient-compression-quantization-sparsification' 1.1:
    stochastic rounding is unbiased in expectation)."""
    bits = 2 if mode == "tern" else 2
    x = np.array([0.1, -0.37, 0.9, 0.55, -1.0, 0.0, 0.2, 0.73], np.float32)
    N = 4000
    acc = np.zeros(x.size)
    acc2 = np.zeros(x.size)
    for seed in range(N):
        codes, scales = oracle.quant(x, bits, 0, mode, "stochastic", seed, 0)
        xh = oracle.dequant(codes, scales, x.size, bits, 0, mode).astype(np.float64)
        acc += xh
        acc2 += xh * xh
    mean = acc / N
    var = acc2 / N - mean ** 2
    sigma = np.sqrt(np.maximum(var, 1e-12))
    assert np.all(np.abs(mean - x) <= 5 * sigma / np.sqrt(N) + 1e-6)


@pytest.mark.parametrize("mode", ["minmax", "qsgd"])
def test_stochastic_codes_bracket_t(mode):
    r = np.random.default_rng(4)
    x = r.standard_normal(4099).astype(np.float32)
    bits, G = 4, 64
    cn, sn = oracle.quant(x, bits, G, mode, "nearest_even")
    cs, ss = oracle.quant(x, bits, G, mode, "stochastic", 123, 7)
    assert np.array_equal(sn, ss)
    mag = (x.size * bits + 7) // 8

    def q_of(c):
        f = np.unpackbits(c[:mag], bitorder="little")[:x.size * bits]
        return (f.reshape(-1, bits) * (1 << np.arange(bits))).sum(axis=1)

    qn, qs = q_of(cn), q_of(cs)
    assert np.all(np.abs(qn - qs) <= 1)
    # repeatable for the same (seed, step); a different step draws anew
    assert np.array_equal(cs, oracle.quant(x, bits, G, mode, "stochastic", 123, 7)[0])
    assert not np.array_equal(cs, oracle.quant(x, bits, G, mode, "stochastic", 123, 8)[0])


def test_tern_properties():
    r = np.random.default_rng(8)
    x = r.standard_normal(1000).astype(np.float32)
    for rounding in ("nearest_even", "stochastic"):
        codes, scales = oracle.quant(x, 2, 0, "tern", rounding, 9, 1)
        xh = oracle.dequant(codes, scales, x.size, 2, 0, "tern")
        s = scales[0]
        assert s == np.abs(x).max()
        assert set(np.unique(xh).tolist()) <= {-s, 0.0, s}
        j = int(np.argmax(np.abs(x)))
        assert xh[j] == x[j]  # the max always maps to +-scale
        assert np.all(np.sign(xh[xh != 0]) == np.sign(x[xh != 0]))


@pytest.mark.parametrize("mode,bits", [("minmax", 8), ("minmax", 4), ("qsgd", 8),
                                       ("qsgd", 2), ("tern", 2)])
def test_error_feedback_identity(mode, bits):
    """e' = fl(c - g_hat): c - g_hat - e' is within half an ulp of e', and
    c = g_hat + e' exactly wherever the subtraction is exact (Sterbenz)."""
    r = np.random.default_rng(bits)
    g = r.standard_normal(3000).astype(np.float32)
    e = (0.01 * r.standard_normal(3000)).astype(np.float32)
    codes, scales, e2 = oracle.ef_quant(g, e, bits, 64, mode, "stochastic", 1, 2)
    xh = oracle.dequant(codes, scales, g.size, bits, 64, mode)
    c = g + e
    diff = c.astype(np.float64) - xh.astype(np.float64) - e2.astype(np.float64)
    assert np.all(np.abs(diff) <= 0.5 * np.spacing(np.abs(e2)) + 1e-45)
    ster = (xh != 0) & (np.sign(xh) == np.sign(c)) & \
        (np.abs(xh) >= np.abs(c) / 2) & (np.abs(xh) <= 2 * np.abs(c))
    assert np.array_equal((xh + e2)[ster], c[ster])


def test_hybrid_composition():
    """EF + Top-K + QSGD equals the composition of the two oracle calls."""
    r = np.random.default_rng(21)
    g = r.standard_normal(5000).astype(np.float32)
    e = (0.1 * r.standard_normal(5000)).astype(np.float32)
    k = 50
    idx, codes, scales, e2 = oracle.ef_topk_quant(g, e, k, 8, 64, "stochastic", 3, 4)
    idx_t, val_t, e_t = oracle.ef_topk(g, e, k)
    codes_q, scales_q = oracle.quant(val_t, 8, 64, "qsgd", "stochastic", 3, 4)
    xh = oracle.dequant(codes_q, scales_q, k, 8, 64, "qsgd")
    assert np.array_equal(idx, idx_t) and np.array_equal(codes, codes_q)
    assert np.array_equal(scales, scales_q)
    want = e_t.copy()
    want[idx_t] = val_t - xh
    assert np.array_equal(e2, want)


def test_rejects_bad_arguments():
    x = np.ones(8, np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.quant(x, 3, 0, "minmax")
    with pytest.raises(oracle.OracleError):
        oracle.quant(x, 4, 0, "tern")


def test_quant_at_matches_full_call():
    """A group-aligned slice quantised with its call offset reproduces the
    corresponding bytes of the full call (what the sampled full-size parity
    tests rely on)."""
    r = np.random.default_rng(31)
    x = r.standard_normal(64 * 40 + 24).astype(np.float32)
    for mode, bits in (("minmax", 4), ("qsgd", 8), ("minmax", 1)):
        full_c, full_s = oracle.quant(x, bits, 64, mode, "stochastic", 5, 6)
        g0, g1 = 7, 23
        c, s = oracle.quant_at(x[g0 * 64:g1 * 64], g0 * 64, bits, 64, mode,
                               "stochastic", 5, 6)
        per = 2 if mode == "minmax" else 1
        assert np.array_equal(s, full_s[g0 * per:g1 * per])
        nb = 64 * bits // 8
        assert np.array_equal(c[:(g1 - g0) * nb], full_c[g0 * nb:g1 * nb])
