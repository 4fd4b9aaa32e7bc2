"""EF + Top-K + QSGD (hybrid) on the GPU against the oracle, bit for bit."""
import numpy as np
import pytest

import oracle
from gradient_compression_ef_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, dev_f32, host, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from gradient_compression_ef_gb300 import gc
    ctx = gc.Context(16_777_216)
    yield torch, gc, ctx
    ctx.close()


def check(env, g, e, k, bits, group, rounding, seed, step, what):
    torch, gc, ctx = env
    gd, ed = dev_f32(torch, g), dev_f32(torch, e)
    idx = torch.full((max(k, 1),), -1, dtype=torch.int32, device="cuda")
    codes = torch.full((max(gc.codes_bytes(k, bits, "qsgd"), 1),), 0x5A, dtype=torch.uint8,
                       device="cuda")
    scales = torch.full((max(gc.scales_floats(k, group, "qsgd"), 1),), -1.0,
                        dtype=torch.float32, device="cuda")
    gc.ef_topk_quant(ctx, gd, ed, k, bits, group, rounding, seed, step, idx, codes, scales)
    ctx.check()
    o_idx, o_codes, o_scales, o_err = oracle.ef_topk_quant(g, e, k, bits, group, rounding,
                                                           seed, step)
    assert_bits_equal(host(idx)[:k], o_idx, what + " idx")
    assert_bits_equal(host(codes)[:o_codes.size], o_codes, what + " codes")
    assert_bits_equal(host(scales)[:o_scales.size], o_scales, what + " scales")
    assert_bits_equal(host(ed), o_err, what + " err")


@pytest.mark.parametrize("n,k", [(1, 1), (5, 3), (4097, 41), (100_003, 1_000), (333_333, 3_333),
                                 (50_000, 50_000)])
@pytest.mark.parametrize("bits", [8, 4, 2])
@pytest.mark.parametrize("rounding", ["nearest_even", "stochastic"])
def test_sizes(env, n, k, bits, rounding):
    r = np.random.default_rng(n + bits)
    g = r.standard_normal(n).astype(np.float32)
    e = (0.2 * r.standard_normal(n)).astype(np.float32)
    check(env, g, e, k, bits, 64, rounding, 5, 9, "n=%d k=%d" % (n, k))


@pytest.mark.parametrize("group", [4, 16, 128])
def test_groups(env, group):
    r = np.random.default_rng(group)
    g = r.standard_normal(77_777).astype(np.float32)
    check(env, g, np.zeros_like(g), 777, 8, group, "stochastic", 1, 2, "group %d" % group)


def test_k_zero_is_pure_error_feedback(env):
    r = np.random.default_rng(3)
    g = r.standard_normal(1000).astype(np.float32)
    e = r.standard_normal(1000).astype(np.float32)
    check(env, g, e, 0, 8, 64, "nearest_even", 0, 0, "k=0")


def test_transformer_tensor_full_size(env):
    """A 4096 x 4096 tensor of the transformer workload, Top-K 1 % then
    8-bit QSGD (groups of 64) on the kept values, stochastic, two EF steps."""
    g1 = inputs.transformer_tensor(0, 0)
    g2 = inputs.transformer_tensor(1, 0)
    n = g1.size
    k = inputs.ratio_k(n, 1, 100)
    torch, gc, ctx = env
    e = np.zeros(n, np.float32)
    ed = dev_f32(torch, e)
    oe = e
    for step, g in enumerate((g1, g2)):
        gd = dev_f32(torch, g)
        idx = torch.empty(k, dtype=torch.int32, device="cuda")
        codes = torch.empty(gc.codes_bytes(k, 8, "qsgd"), dtype=torch.uint8, device="cuda")
        scales = torch.empty(gc.scales_floats(k, 64, "qsgd"), dtype=torch.float32, device="cuda")
        gc.ef_topk_quant(ctx, gd, ed, k, 8, 64, "stochastic", 42, step, idx, codes, scales)
        ctx.check()
        o_idx, o_codes, o_scales, oe = oracle.ef_topk_quant(g, oe, k, 8, 64, "stochastic", 42,
                                                            step)
        assert_bits_equal(host(idx), o_idx, "step %d idx" % step)
        assert_bits_equal(host(codes), o_codes, "step %d codes" % step)
        assert_bits_equal(host(scales), o_scales, "step %d scales" % step)
        assert_bits_equal(host(ed), oe, "step %d err" % step)


def test_unsupported_group_rejected_before_work(env):
    torch, gc, ctx = env
    g = torch.ones(1000, dtype=torch.float32, device="cuda")
    e = torch.zeros(1000, dtype=torch.float32, device="cuda")
    idx = torch.zeros(16, dtype=torch.int32, device="cuda")
    codes = torch.zeros(64, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(gc.GCError) as ei:
        gc.ef_topk_quant(ctx, g, e, 10, 8, 100, "nearest_even", 0, 0, idx, codes, scales)
    assert ei.value.status == gc.ERR_UNSUPPORTED
    assert float(e.abs().sum()) == 0.0  # nothing ran
