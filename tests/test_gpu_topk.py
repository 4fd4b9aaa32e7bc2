"""EF + Top-K on the GPU against the oracle, bit for bit: indices, values
and residuals, on edge cases, several tiles with ragged tails, ties, the
Python demo's two steps and buckets of the 512 MiB correlated workload."""
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
    ctx = gc.Context(8_000_000)
    yield torch, gc, ctx
    ctx.close()


def run_topk(env, g, e, k):
    torch, gc, ctx = env
    n = g.size
    gd = dev_f32(torch, g)
    ed = dev_f32(torch, e) if e is not None else None
    idx = torch.full((max(k, 1),), -7, dtype=torch.int32, device="cuda")
    val = torch.full((max(k, 1),), -7.0, dtype=torch.float32, device="cuda")
    gc.ef_topk(ctx, gd, ed, k, idx, val)
    ctx.check()
    return host(idx)[:k], host(val)[:k], (host(ed) if ed is not None else None)


def check(env, g, e, k, what):
    idx, val, err = run_topk(env, g, e, k)
    o_idx, o_val, o_err = oracle.ef_topk(g, e, k)
    assert_bits_equal(idx, o_idx, what + " idx")
    assert_bits_equal(val, o_val, what + " val")
    if e is not None:
        assert_bits_equal(err, o_err, what + " err")


@pytest.mark.parametrize("name,x", inputs.tiny_cases(), ids=[c[0] for c in inputs.tiny_cases()])
def test_edge_cases(env, name, x):
    r = np.random.default_rng(len(x))
    e = (0.25 * r.standard_normal(x.size)).astype(np.float32)
    n = x.size
    for k in sorted({0, 1, n // 7, max(n - 1, 0), n}):
        check(env, x, e, k, "%s k=%d ef" % (name, k))
        check(env, x, None, k, "%s k=%d plain" % (name, k))


@pytest.mark.parametrize("n", [2048 * 3 + 17, 100_000, 1_000_003])
@pytest.mark.parametrize("per_mille", [10, 1])
def test_random_sizes(env, n, per_mille):
    r = np.random.default_rng(n + per_mille)
    g = r.standard_normal(n).astype(np.float32)
    e = (0.3 * r.standard_normal(n)).astype(np.float32)
    check(env, g, e, inputs.ratio_k(n, per_mille, 1000), "n=%d" % n)


def test_heavy_ties(env):
    r = np.random.default_rng(5)
    n = 300_001
    g = (r.integers(-6, 7, size=n) * 0.125).astype(np.float32)
    e = np.zeros(n, np.float32)
    for k in (1, 777, 50_000, 123_457):
        check(env, g, e, k, "ties k=%d" % k)


def test_many_candidates_in_one_bin(env):
    """All values in one 12-bit bin: the refinement handles n candidates."""
    r = np.random.default_rng(6)
    n = 200_000
    g = (1.0 + r.integers(0, 1 << 19, size=n) * 2.0 ** -23).astype(np.float32)
    g *= r.choice([-1.0, 1.0], size=n).astype(np.float32)
    check(env, g, np.zeros(n, np.float32), 2_000, "one bin")


def test_demo_two_steps(env):
    g = inputs.demo_gradient()
    k = inputs.ratio_k(g.size, 1, 100)
    e0 = np.zeros_like(g)
    idx1, val1, e1 = run_topk(env, g, e0, k)
    o1 = oracle.ef_topk(g, e0, k)
    assert_bits_equal(idx1, o1[0], "step1 idx")
    assert_bits_equal(e1, o1[2], "step1 err")
    g2 = g * np.float32(0.9)
    idx2, val2, e2 = run_topk(env, g2, e1, k)
    o2 = oracle.ef_topk(g2, o1[2], k)
    assert_bits_equal(idx2, o2[0], "step2 idx")
    assert_bits_equal(val2, o2[1], "step2 val")
    assert_bits_equal(e2, o2[2], "step2 err")


def test_correlated_buckets_full_size(env):
    """Buckets of the 134,217,728-element workload (first, middle and the
    partial last bucket), two correlated EF steps, k = 1 % and 0.1 %."""
    bounds = inputs.bucket_bounds()
    picks = [bounds[0], bounds[10], bounds[-1]]
    r = inputs.rng(99)
    for start, length in picks:
        g1 = inputs.student_t(r, length)
        g2 = (g1 * np.float32(0.9) + inputs.student_t(r, length) * np.float32(0.436))
        g2 = g2.astype(np.float32)
        for per_mille in (10, 1):
            k = inputs.ratio_k(length, per_mille, 1000)
            e = np.zeros(length, np.float32)
            oe = e.copy()
            for step, g in enumerate((g1, g2)):
                idx, val, e = run_topk(env, g, e, k)
                o_idx, o_val, oe = oracle.ef_topk(g, oe, k)
                what = "bucket@%d k=%d step%d" % (start, k, step)
                assert_bits_equal(idx, o_idx, what + " idx")
                assert_bits_equal(val, o_val, what + " val")
                assert_bits_equal(e, oe, what + " err")


def test_contexts_on_streams_agree(env):
    """Buckets on several contexts / streams give the sequential results."""
    torch, gc, _ = env
    r = np.random.default_rng(12)
    n, nb, k = 400_000, 6, 4_000
    gs = [r.standard_normal(n).astype(np.float32) for _ in range(nb)]
    streams = [torch.cuda.Stream() for _ in range(3)]
    ctxs = [gc.Context(n, stream=s) for s in streams]
    outs = []
    for b in range(nb):
        s = streams[b % 3]
        with torch.cuda.stream(s):
            gd = dev_f32(torch, gs[b])
            ed = torch.zeros(n, dtype=torch.float32, device="cuda")
            idx = torch.empty(k, dtype=torch.int32, device="cuda")
            val = torch.empty(k, dtype=torch.float32, device="cuda")
        gc.ef_topk(ctxs[b % 3], gd, ed, k, idx, val)
        outs.append((idx, val, ed))
    for c in ctxs:
        c.check()
        c.close()
    for b in range(nb):
        o = oracle.ef_topk(gs[b], np.zeros(n, np.float32), k)
        assert_bits_equal(host(outs[b][0]), o[0], "stream idx")
        assert_bits_equal(host(outs[b][2]), o[2], "stream err")


def test_rejects_bad_arguments(env):
    torch, gc, ctx = env
    g = torch.zeros(1025, dtype=torch.float32, device="cuda")
    idx = torch.zeros(8, dtype=torch.int32, device="cuda")
    val = torch.zeros(8, dtype=torch.float32, device="cuda")
    with pytest.raises(gc.GCError) as ei:
        gc.ef_topk(ctx, g[1:], None, 4, idx, val, n=1024)
    assert ei.value.status == gc.ERR_ALIGNMENT
    with pytest.raises(gc.GCError) as ei:
        gc.ef_topk(ctx, g, None, 2000, idx, val)
    assert ei.value.status == gc.ERR_INVALID_ARG
    small = gc.Context(100)
    with pytest.raises(gc.GCError) as ei:
        gc.ef_topk(small, g, None, 4, idx, val)
    assert ei.value.status == gc.ERR_WORKSPACE
    small.close()
