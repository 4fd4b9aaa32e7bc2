"""Quantisation, packing, dequantisation and EF residual on the GPU against
the oracle, bit for bit (codes including padding, scales, residuals), for
every mode, bit width, rounding, fused and multi-pass group sizes, edge
cases, and sampled group ranges of the 2^30-element workload."""
import numpy as np
import pytest

import oracle
from gradient_compression_ef_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, dev_f32, host, torch_cuda

pytestmark = pytest.mark.gpu

MODE_BITS = [("minmax", 1), ("minmax", 2), ("minmax", 4), ("minmax", 8),
             ("qsgd", 1), ("qsgd", 2), ("qsgd", 4), ("qsgd", 8), ("tern", 2)]


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from gradient_compression_ef_gb300 import gc
    ctx = gc.Context(2_000_000)
    yield torch, gc, ctx
    ctx.close()


def gpu_quant(env, x, e, bits, group, mode, rounding, seed, step):
    torch, gc, ctx = env
    n = x.size
    xd = dev_f32(torch, x)
    codes = torch.full((max(gc.codes_bytes(n, bits, mode), 1),), 0xA5, dtype=torch.uint8,
                       device="cuda")
    scales = torch.full((max(gc.scales_floats(n, group, mode), 1),), -3.0,
                        dtype=torch.float32, device="cuda")
    ed = None
    if e is None:
        gc.quant(ctx, xd, bits, group, mode, rounding, seed, step, codes, scales)
    else:
        ed = dev_f32(torch, e)
        gc.ef_quant(ctx, xd, ed, bits, group, mode, rounding, seed, step, codes, scales)
    ctx.check()
    nb = gc.codes_bytes(n, bits, mode)
    ns = gc.scales_floats(n, group, mode)
    return (host(codes)[:nb], host(scales)[:ns], host(ed) if ed is not None else None,
            codes, scales)


def gpu_dequant(env, codes, scales, n, bits, group, mode):
    torch, gc, ctx = env
    out = torch.full((max(n, 1),), 9.0, dtype=torch.float32, device="cuda")
    gc.dequant(ctx, codes, scales, n, bits, group, mode, out)
    ctx.check()
    return host(out)[:n]


def check(env, x, e, bits, group, mode, rounding, seed=3, step=5, what=""):
    c, s, err, cd, sd = gpu_quant(env, x, e, bits, group, mode, rounding, seed, step)
    if e is None:
        oc, os_ = oracle.quant(x, bits, group, mode, rounding, seed, step)
    else:
        oc, os_, oe = oracle.ef_quant(x, e, bits, group, mode, rounding, seed, step)
        assert_bits_equal(err, oe, what + " err")
    assert_bits_equal(c, oc, what + " codes")
    assert_bits_equal(s, os_, what + " scales")
    xh = gpu_dequant(env, cd, sd, x.size, bits, group, mode)
    assert_bits_equal(xh, oracle.dequant(oc, os_, x.size, bits, group, mode), what + " dequant")


@pytest.mark.parametrize("mode,bits", MODE_BITS)
@pytest.mark.parametrize("group", [4, 32, 64, 128, 3, 100, 1000, 5000, 0])
@pytest.mark.parametrize("rounding", ["nearest_even", "stochastic"])
def test_modes_groups(env, mode, bits, group, rounding):
    r = np.random.default_rng(bits * 1000 + group)
    n = 20_011
    x = (0.01 * r.standard_normal(n)).astype(np.float32)
    x[r.integers(0, n, 20)] *= 100
    e = (0.001 * r.standard_normal(n)).astype(np.float32)
    check(env, x, None, bits, group, mode, rounding, what="plain")
    check(env, x, e, bits, group, mode, rounding, what="ef")


@pytest.mark.parametrize("name,x", inputs.tiny_cases(), ids=[c[0] for c in inputs.tiny_cases()])
@pytest.mark.parametrize("mode,bits", [("minmax", 8), ("minmax", 1), ("qsgd", 4), ("tern", 2)])
def test_edge_cases(env, name, x, mode, bits):
    for group in (4, 64, 7, 0):
        for rounding in ("nearest_even", "stochastic"):
            check(env, x, np.zeros_like(x), bits, group, mode, rounding,
                  what="%s g=%d %s" % (name, group, rounding))


def test_demo_whole_tensor_minmax8(env):
    """The demo's quantize(grad, 8): one min-max group over 10^6 values."""
    g = inputs.demo_gradient()
    check(env, g, None, 8, 0, "minmax", "nearest_even", what="demo")


def test_group64_full_size_sampled(env):
    """The 2^30-element outlier workload, groups of 64, with EF; sampled
    group ranges (start, middle, end) checked against the oracle."""
    torch, gc, ctx = env
    n = inputs.GROUP_ELEMS
    x = inputs.outlier_gradient(n)
    e = (1e-3 * inputs.rng(8).standard_normal(n, dtype=np.float32)).astype(np.float32)
    big = gc.Context(1024)  # the fused kernel needs no scratch
    xd, ed0 = dev_f32(torch, x), dev_f32(torch, e)
    G = 64
    ranges = [(0, 512), (n // G // 2, n // G // 2 + 512), (n // G - 512, n // G)]
    for mode, bits in (("minmax", 8), ("minmax", 4), ("qsgd", 8), ("qsgd", 4)):
        for rounding in ("nearest_even", "stochastic"):
            ed = ed0.clone()
            codes = torch.empty(gc.codes_bytes(n, bits, mode), dtype=torch.uint8, device="cuda")
            scales = torch.empty(gc.scales_floats(n, G, mode), dtype=torch.float32,
                                 device="cuda")
            gc.ef_quant(big, xd, ed, bits, G, mode, rounding, 17, 2, codes, scales)
            big.check()
            mag = (n * bits + 7) // 8
            for g0, g1 in ranges:
                a, b = g0 * G, g1 * G
                c = x[a:b] + e[a:b]
                oc, os_ = oracle.quant_at(c, a, bits, G, mode, rounding, 17, 2)
                per = 2 if mode == "minmax" else 1
                what = "%s%d %s groups %d..%d" % (mode, bits, rounding, g0, g1)
                assert_bits_equal(host(scales[g0 * per:g1 * per]), os_, what + " scales")
                nb = (b - a) * bits // 8
                assert_bits_equal(host(codes[a * bits // 8:a * bits // 8 + nb]), oc[:nb],
                                  what + " codes")
                if mode == "qsgd":
                    sb = (mag + 15) // 16 * 16
                    s_o = oc[(nb + 15) // 16 * 16:][:(b - a) // 8]
                    assert_bits_equal(host(codes[sb + a // 8:sb + b // 8]), s_o, what + " signs")
                xh = oracle.dequant(oc, os_, b - a, bits, G, mode)
                assert_bits_equal(host(ed[a:b]), c - xh, what + " err")
            del codes, scales, ed
    big.close()


def test_terngrad_layer_tensors(env):
    """Layer-wise TernGrad (one scale per tensor), stochastic, with EF, on
    the 4096 x 11008 and 4096 tensors of the transformer workload."""
    torch, gc, _ = env
    big = gc.Context(45_088_768)
    for which in (4, 7):
        x = inputs.transformer_tensor(3, which)
        e = (0.3 * inputs.transformer_tensor(4, which)).astype(np.float32)
        torch_ctx = (torch, gc, big)
        check(torch_ctx, x, e, 2, 0, "tern", "stochastic", seed=3 * 1000 + which, step=1,
              what="tern tensor %d" % which)
    big.close()


def test_rejects_bad_arguments(env):
    torch, gc, ctx = env
    x = torch.zeros(1000, dtype=torch.float32, device="cuda")
    codes = torch.zeros(2000, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(100, dtype=torch.float32, device="cuda")
    for bits, mode, status in ((3, "minmax", gc.ERR_UNSUPPORTED), (4, "tern", gc.ERR_UNSUPPORTED)):
        with pytest.raises(gc.GCError) as ei:
            gc.quant(ctx, x, bits, 64, mode, "nearest_even", 0, 0, codes, scales)
        assert ei.value.status == status
    with pytest.raises(gc.GCError) as ei:
        gc.quant(ctx, x[1:], 8, 64, "minmax", "nearest_even", 0, 0, codes, scales, n=999)
    assert ei.value.status == gc.ERR_ALIGNMENT
    small = gc.Context(10)
    with pytest.raises(gc.GCError) as ei:  # multi-pass groups need scratch
        gc.quant(small, x, 8, 100, "minmax", "nearest_even", 0, 0, codes, scales)
    assert ei.value.status == gc.ERR_WORKSPACE
    gc.quant(small, x, 8, 64, "minmax", "nearest_even", 0, 0, codes, scales)  # fused: fine
    small.check()
    small.close()
