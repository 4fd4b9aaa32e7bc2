"""Logarithmic and differential quantisation on the GPU against the oracle,
bit for bit ('分布式训练中的梯度压缩算法' 二.1 对数量化, 二.4 差分量化):
codes with padding, scales, residuals, histories and the receiver's
reconstruction, for every bit width, rounding, fused and multi-pass group
sizes, ragged sizes and several error-feedback steps."""
import numpy as np
import pytest

import oracle
from gradient_compression_ef_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, dev_f32, host, torch_cuda
from tests.test_gpu_quant import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from gradient_compression_ef_gb300 import gc
    ctx = gc.Context(2_000_000)
    yield torch, gc, ctx
    ctx.close()


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("group", [4, 64, 128, 3, 1000, 0])
@pytest.mark.parametrize("rounding", ["nearest_even", "stochastic"])
def test_log_modes_groups(env, bits, group, rounding):
    r = np.random.default_rng(bits * 100 + group)
    n = 20_011
    x = (r.standard_normal(n) * 3).astype(np.float32)
    x[r.integers(0, n, 20)] *= 1000
    x[r.integers(0, n, 20)] = 0.0
    e = (0.01 * r.standard_normal(n)).astype(np.float32)
    check(env, x, None, bits, group, "log", rounding, what="log plain")
    check(env, x, e, bits, group, "log", rounding, what="log ef")


@pytest.mark.parametrize("n", [1, 5, 128, 4097, 100_003])
def test_log_ragged(env, n):
    r = np.random.default_rng(n)
    x = (r.standard_normal(n) * 1e-3).astype(np.float32)
    check(env, x, np.zeros_like(x), 8, 64, "log", "stochastic", what="ragged")


def test_log_extremes(env):
    """Magnitudes over the whole binary32 range, zero groups and ties."""
    x = np.array([0.0] * 64 + [3.0e38, -1e-30, 1e-45, -2.0] * 16 + [1.5] * 64, np.float32)
    for group in (64, 0):
        check(env, x, None, 4, group, "log", "nearest_even", what="extremes")


def test_log_rejects_one_bit(env):
    torch, gc, ctx = env
    x = torch.zeros(64, device="cuda")
    c = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(gc.GCError) as ex:
        gc.quant(ctx, x, 1, 64, "log", "nearest_even", 0, 0, c, x)
    assert ex.value.status == gc.ERR_UNSUPPORTED


def run_diff(env, g, e, ref, bits, group, mode, rounding, seed, step, refresh):
    torch, gc, ctx = env
    n = g.size
    gd = dev_f32(torch, g)
    ed = dev_f32(torch, e) if e is not None else None
    rd = dev_f32(torch, ref)
    codes = torch.full((max(gc.codes_bytes(n, bits, mode), 1),), 0xA5, dtype=torch.uint8,
                       device="cuda")
    scales = torch.full((max(gc.scales_floats(n, group, mode), 1),), -3.0,
                        dtype=torch.float32, device="cuda")
    gc.ef_diff_quant(ctx, gd, ed, rd, bits, group, mode, rounding, seed, step, refresh, codes,
                     scales)
    ctx.check()
    nb, ns = gc.codes_bytes(n, bits, mode), gc.scales_floats(n, group, mode)
    return (host(codes)[:nb], host(scales)[:ns], host(ed) if ed is not None else None,
            host(rd), codes, scales)


DIFF_MODES = [("minmax", 4), ("minmax", 1), ("qsgd", 8), ("qsgd", 2), ("tern", 2), ("log", 8),
              ("log", 4)]


@pytest.mark.parametrize("mode,bits", DIFF_MODES)
@pytest.mark.parametrize("group", [4, 32, 128])
@pytest.mark.parametrize("ef", [True, False])
def test_diff_steps(env, mode, bits, group, ef):
    """Five correlated steps, a refresh at step 0 and 3: codes, scales,
    residual and history equal the oracle's; the receiver's history equals
    the sender's."""
    torch, gc, ctx = env
    n = 10_007
    r = np.random.default_rng(bits + group)
    g = r.standard_normal(n).astype(np.float32)
    e = np.zeros(n, np.float32) if ef else None
    ref = np.zeros(n, np.float32)
    recv = torch.zeros(n, dtype=torch.float32, device="cuda")
    for step in range(5):
        g = (0.9 * g + 0.3 * r.standard_normal(n)).astype(np.float32)
        refresh = step in (0, 3)
        c, s, e2, ref2, cd, sd = run_diff(env, g, e, ref, bits, group, mode, "stochastic", 7,
                                          step, refresh)
        oc, os_, oe, oref = oracle.ef_diff_quant(g, e, ref, bits, group, mode, "stochastic", 7,
                                                 step, refresh)
        w = "%s/%d g%d step %d" % (mode, bits, group, step)
        assert_bits_equal(c, oc, w + " codes")
        assert_bits_equal(s, os_, w + " scales")
        assert_bits_equal(ref2, oref, w + " ref")
        if ef:
            assert_bits_equal(e2, oe, w + " err")
            e = oe
        ref = oref
        gc.diff_dequant(ctx, cd, sd, n, bits, group, mode, refresh, recv)
        ctx.check()
        assert_bits_equal(host(recv), oref, w + " receiver")


def test_diff_validation(env):
    torch, gc, ctx = env
    x = torch.zeros(256, device="cuda")
    c = torch.zeros(256, dtype=torch.uint8, device="cuda")
    for group in (0, 3, 256, 1000):
        with pytest.raises(gc.GCError) as ex:
            gc.ef_diff_quant(ctx, x, x, x, 8, group, "qsgd", "nearest_even", 0, 0, False, c, x)
        assert ex.value.status == gc.ERR_UNSUPPORTED
    with pytest.raises(gc.GCError) as ex:
        gc.ef_diff_quant(ctx, x, x, None, 8, 64, "qsgd", "nearest_even", 0, 0, False, c, x)
    assert ex.value.status == gc.ERR_INVALID_ARG


def test_full_size_log_and_diff(env):
    """The 134,217,728-element gradient: 8-bit logarithmic quantisation in
    groups of 64 and two steps of 4-bit min-max differential quantisation
    (nearest-even, so a group-aligned slice is an independent problem);
    sampled slices against the oracle."""
    torch, gc, _ = env
    n = inputs.FLAT_ELEMS
    ctx = gc.Context(0)
    g = inputs.student_t_device(n, "cuda", seed=31)
    e = torch.zeros(n, dtype=torch.float32, device="cuda")
    ref = torch.zeros(n, dtype=torch.float32, device="cuda")
    codes = torch.empty(gc.codes_bytes(n, 8, "log"), dtype=torch.uint8, device="cuda")
    scales = torch.empty(gc.scales_floats(n, 64, "log"), dtype=torch.float32, device="cuda")
    gc.ef_quant(ctx, g, e, 8, 64, "log", "nearest_even", 0, 0, codes, scales)
    ctx.check()
    gh = host(g)
    for s0 in (0, n // 2 + 64 * 1001, n - 64 * 300):
        sl = slice(s0, s0 + 64 * 300)
        oc, os_, oe = oracle.ef_quant(gh[sl], np.zeros(64 * 300, np.float32), 8, 64, "log")
        assert_bits_equal(host(codes[s0:s0 + 64 * 300]), oc, "log codes @%d" % s0)
        assert_bits_equal(host(scales[s0 // 64:s0 // 64 + 300]), os_, "log scales @%d" % s0)
        assert_bits_equal(host(e[sl]), oe, "log err @%d" % s0)
    e.zero_()
    codes4 = torch.empty(gc.codes_bytes(n, 4, "minmax"), dtype=torch.uint8, device="cuda")
    scales4 = torch.empty(gc.scales_floats(n, 64, "minmax"), dtype=torch.float32, device="cuda")
    ref_h, e_h = np.zeros(0, np.float32), None
    g2 = g
    for step in range(2):
        if step == 1:
            g2 = (g * 0.9).contiguous()
            ref_h, e_h = host(ref), host(e)
        gc.ef_diff_quant(ctx, g2, e, ref, 4, 64, "minmax", "nearest_even", 0, step, step == 0,
                         codes4, scales4)
    ctx.check()
    g2h = host(g2)
    for s0 in (64 * 7, n - 64 * 500):
        sl = slice(s0, s0 + 64 * 500)
        oc, os_, oe, oref = oracle.ef_diff_quant(g2h[sl], e_h[sl], ref_h[sl], 4, 64, "minmax")
        assert_bits_equal(host(codes4[s0 // 2:(s0 + 64 * 500) // 2]), oc[:64 * 500 // 2],
                          "diff codes @%d" % s0)
        assert_bits_equal(host(scales4[s0 // 32:s0 // 32 + 1000]), os_, "diff scales @%d" % s0)
        assert_bits_equal(host(e[sl]), oe, "diff err @%d" % s0)
        assert_bits_equal(host(ref[sl]), oref, "diff ref @%d" % s0)
    ctx.close()
