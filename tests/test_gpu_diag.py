"""Fused per-bucket diagnostics of the bucketed calls against the oracle
('gradient-compression-quantization-sparsification' 3.2: gradient norm
ratio; '梯度聚合通信优化实战方案' Python 演示: error energy).

Tolerance: every GPU sum is of non-negative terms, accumulated in binary32
by fused multiply-add in runs of at most 64 terms per lane, added over the
32 lanes of a warp (5 more roundings), combined from at most three passes
(2 more) into one binary32 partial per segment or chunk, and the partials
summed per bucket by compensated summation (about 2 roundings); its
relative error is at most 73 * 2^-24 < 4.4e-6 of the exact sum, and the
oracle's binary64 sums are exact to about 1e-9, so the test allows 1e-5
relative.  A value whose exact sum is 0 must be exactly 0."""
import numpy as np
import pytest

import oracle
from gradient_compression_ef_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, dev_f32, host, torch_cuda
from tests.test_gpu_buckets import LAYOUTS, make_inputs, many_buckets, starts

pytestmark = pytest.mark.gpu

RTOL = 1e-5


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from gradient_compression_ef_gb300 import gc
    ctx = gc.Context(8_000_000)
    yield torch, gc, ctx
    ctx.close()


def assert_diag(got, want, what):
    for q in range(3):
        g, w = float(got[q]), float(want[q])
        if w == 0.0:
            assert g == 0.0, "%s [%d]: %r, want 0" % (what, q, g)
        else:
            assert abs(g - w) <= RTOL * w, "%s [%d]: %r vs %r" % (what, q, g, w)


def run_topk(env, ns, ks, gd, ed):
    torch, gc, ctx = env
    oi, _, _ = gc.bucket_offsets(ks)
    idx = torch.full((max(oi[-1], 4),), -7, dtype=torch.int32, device="cuda")
    val = torch.full((max(oi[-1], 4),), -7.0, dtype=torch.float32, device="cuda")
    diag = torch.full((3 * len(ns),), -1.0, dtype=torch.float64, device="cuda")
    gc.ef_topk_buckets(ctx, gd, ed, idx, val, diag=diag)
    ctx.check()
    return oi, host(idx), host(val), host(diag)


def check_topk(ns, ks, g, e, oi, idx, val, diag, what, err=None):
    st = starts(ns)
    for b, (n, k) in enumerate(zip(ns, ks)):
        sl = slice(st[b], st[b + 1])
        eb = None if e is None else e[sl]
        o_idx, o_val, o_err = oracle.ef_topk(g[sl], None if eb is None else eb.copy(), k)
        w = "%s bucket %d" % (what, b)
        assert_bits_equal(idx[oi[b]:oi[b] + k], o_idx, w + " idx")
        assert_bits_equal(val[oi[b]:oi[b] + k], o_val, w + " val")
        if err is not None:
            assert_bits_equal(err[sl], o_err, w + " err")
        assert_diag(diag[3 * b:3 * b + 3], oracle.diagnostics(g[sl], eb, o_idx, o_val), w)


@pytest.mark.parametrize("name", sorted(LAYOUTS))
@pytest.mark.parametrize("ef", [True, False])
def test_topk_layouts(env, name, ef):
    torch, gc, ctx = env
    ns, ks = LAYOUTS[name]
    g, e = make_inputs(ns, 3 + len(name))
    e = e if ef else None
    ctx.set_buckets(ns, ks)
    ed = dev_f32(torch, e) if ef else None
    oi, idx, val, diag = run_topk(env, ns, ks, dev_f32(torch, g), ed)
    check_topk(ns, ks, g, e, oi, idx, val, diag, name, host(ed) if ef else None)


def test_topk_many_buckets(env):
    torch, gc, ctx = env
    ns, ks = many_buckets(12)
    g, e = make_inputs(ns, 12)
    ctx.set_buckets(ns, ks)
    oi, idx, val, diag = run_topk(env, ns, ks, dev_f32(torch, g), dev_f32(torch, e))
    check_topk(ns, ks, g, e, oi, idx, val, diag, "many")


@pytest.mark.parametrize("scales", [(1.0, 1.0, 1.0), (1.0, 0.25, 4.0, 16.0, 0.01)])
def test_topk_threshold_reuse_paths(env, scales):
    """Correlated steps whose magnitudes jump: later calls select from the
    lists of the previous threshold's guess, or fall back to re-reading c;
    the diagnostics are right on both paths."""
    torch, gc, ctx = env
    ns, ks = [300_000, 65_536, 100_004, 2_048], [3_000, 655, 10_000, 20]
    n = sum(ns)
    ctx.set_buckets(ns, ks)
    grads = inputs.correlated_steps(n, len(scales), seed=17)
    ed = torch.zeros(n, dtype=torch.float32, device="cuda")
    for step, (gs, f) in enumerate(zip(grads, scales)):
        g = (gs * np.float32(f)).astype(np.float32)
        e_before = host(ed)
        oi, idx, val, diag = run_topk(env, ns, ks, dev_f32(torch, g), ed)
        check_topk(ns, ks, g, e_before, oi, idx, val, diag, "step %d" % step, host(ed))


def run_quant(env, ns, ks, gd, ed, bits, group, rounding, seed, step):
    torch, gc, ctx = env
    oi, oc, os_ = gc.bucket_offsets(ks, bits, group)
    idx = torch.full((max(oi[-1], 4),), -7, dtype=torch.int32, device="cuda")
    codes = torch.full((max(oc[-1], 16),), 0x5A, dtype=torch.uint8, device="cuda")
    scales = torch.full((max(os_[-1], 4),), -1.0, dtype=torch.float32, device="cuda")
    diag = torch.full((3 * len(ns),), -1.0, dtype=torch.float64, device="cuda")
    gc.ef_topk_quant_buckets(ctx, gd, ed, bits, group, rounding, seed, step, idx, codes, scales,
                             diag=diag)
    ctx.check()
    return (oi, oc, os_), host(idx), host(codes), host(diag)


def check_quant(ns, ks, g, e, bits, group, rounding, seed, step, offs, idx, codes, diag, what,
                buckets=None):
    oi, oc, _ = offs
    st = starts(ns)
    for b in (range(len(ns)) if buckets is None else buckets):
        k = ks[b]
        sl = slice(st[b], st[b + 1])
        o_idx, o_codes, o_scales, _ = oracle.ef_topk_quant(
            g[sl], e[sl].copy(), k, bits, group, rounding, oracle.bucket_seed(seed, b), step)
        w = "%s bucket %d" % (what, b)
        assert_bits_equal(idx[oi[b]:oi[b] + k], o_idx, w + " idx")
        assert_bits_equal(codes[oc[b]:oc[b + 1]], o_codes, w + " codes")
        g_hat = oracle.dequant(o_codes, o_scales, k, bits, group, "qsgd")
        assert_diag(diag[3 * b:3 * b + 3], oracle.diagnostics(g[sl], e[sl], o_idx, g_hat), w)


@pytest.mark.parametrize("name", ["tiny", "segments", "mixed", "single"])
@pytest.mark.parametrize("bits,rounding", [(8, "stochastic"), (2, "nearest_even")])
def test_quant_layouts(env, name, bits, rounding):
    torch, gc, ctx = env
    ns, ks = LAYOUTS[name]
    g, e = make_inputs(ns, 40 + bits)
    ctx.set_buckets(ns, ks)
    out = run_quant(env, ns, ks, dev_f32(torch, g), dev_f32(torch, e), bits, 64, rounding, 3, 1)
    check_quant(ns, ks, g, e, bits, 64, rounding, 3, 1, *out, name)


def test_quant_many_buckets_two_steps(env):
    torch, gc, ctx = env
    ns, ks = many_buckets(13, nb=150)
    n = sum(ns)
    ctx.set_buckets(ns, ks)
    grads = inputs.correlated_steps(n, 2, seed=13)
    ed = torch.zeros(n, dtype=torch.float32, device="cuda")
    for step, g in enumerate(grads):
        e_before = host(ed)
        out = run_quant(env, ns, ks, dev_f32(torch, g), ed, 4, 16, "stochastic", 77, step)
        check_quant(ns, ks, g, e_before, 4, 16, "stochastic", 77, step, *out, "step %d" % step)


def test_diagnostics_leave_results_unchanged(env):
    """The same call with and without diagnostics gives identical outputs."""
    torch, gc, ctx = env
    ns, ks = LAYOUTS["mixed"]
    g, e = make_inputs(ns, 8)
    ctx.set_buckets(ns, ks)
    oi, oc, os_ = gc.bucket_offsets(ks, 8, 64)
    res = []
    for with_diag in (False, True):
        ed = dev_f32(torch, e)
        idx = torch.zeros(oi[-1], dtype=torch.int32, device="cuda")
        codes = torch.zeros(oc[-1], dtype=torch.uint8, device="cuda")
        scales = torch.zeros(os_[-1], dtype=torch.float32, device="cuda")
        diag = torch.zeros(3 * len(ns), dtype=torch.float64, device="cuda") if with_diag else None
        gc.ef_topk_quant_buckets(ctx, dev_f32(torch, g), ed, 8, 64, "stochastic", 9, 2, idx,
                                 codes, scales, diag=diag)
        ctx.check()
        res.append((host(ed), host(idx), host(codes), host(scales)))
    for a, b, what in zip(res[0], res[1], ("err", "idx", "codes", "scales")):
        assert_bits_equal(b, a, what)


def test_norm_ratio_limits(env):
    """Everything sent: ratio 1 and no error energy; nothing sent: ratio 0
    and the error energy is the gradient's."""
    torch, gc, ctx = env
    ns, ks = [4096, 4096], [4096, 0]
    g, _ = make_inputs(ns, 1)
    ctx.set_buckets(ns, ks)
    _, _, _, diag = run_topk(env, ns, ks, dev_f32(torch, g), None)
    d = diag.reshape(-1, 3)
    assert abs(np.sqrt(d[0, 1] / d[0, 0]) - 1.0) <= RTOL and d[0, 2] == 0.0
    assert d[1, 1] == 0.0 and d[1, 2] == d[1, 0]


def test_validation(env):
    torch, gc, ctx = env
    ctx.set_buckets([64], [4])
    x = torch.zeros(64, device="cuda")
    i = torch.zeros(64, dtype=torch.int32, device="cuda")
    d = torch.zeros(8, dtype=torch.float64, device="cuda")
    with pytest.raises(gc.GCError) as ex:
        gc.ef_topk_buckets(ctx, x, x, i, x, diag=d[1:])
    assert ex.value.status == gc.ERR_ALIGNMENT


def test_full_size_workload(env):
    """The 134,217,728-element gradient in 21 buckets of 25 MiB, Top-K 1 % +
    8-bit QSGD (groups of 64, stochastic), two correlated EF steps with
    diagnostics: the first, a middle and the last bucket against the oracle
    at the second step."""
    torch, gc, _ = env
    n = inputs.FLAT_ELEMS
    bounds = inputs.bucket_bounds(n)
    ns = [length for _, length in bounds]
    ks = [inputs.ratio_k(length, 10, 1000) for length in ns]
    ctx = gc.Context(max(ns))
    ctx.set_buckets(ns, ks)
    grads = inputs.correlated_steps_device(n, 2, "cuda", seed=6)
    ed = torch.zeros(n, dtype=torch.float32, device="cuda")
    for step, gd in enumerate(grads):
        e_before = host(ed) if step == 1 else None
        out = run_quant((torch, gc, ctx), ns, ks, gd, ed, 8, 64, "stochastic", 2000, step)
    check_quant(ns, ks, host(grads[1]), e_before, 8, 64, "stochastic", 2000, 1, *out, "full",
                buckets=[0, len(ns) // 2, len(ns) - 1])
    ctx.close()
