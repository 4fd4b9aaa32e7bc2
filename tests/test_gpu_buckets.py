"""Bucketed calls (one launch per pass over every bucket of a flat gradient)
on the GPU: each bucket against the oracle bit for bit, and against the
single-bucket entry points at the full-size workload."""
import numpy as np
import pytest

import oracle
from gradient_compression_ef_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, dev_f32, host, torch_cuda

pytestmark = pytest.mark.gpu

# (bucket sizes, kept per bucket): ragged segments, k = 0, k = n, tiny
# buckets, one bucket, sizes around the 2048-element segment
LAYOUTS = {
    "tiny": ([8, 12, 5], [1, 12, 0]),
    "segments": ([4096, 2048, 2044, 6001], [41, 2048, 1, 600]),
    "mixed": ([100_000, 4, 200_004, 33_333], [1_000, 2, 2_000, 333]),
    "single": ([50_001], [500]),
    "one_element": ([1], [1]),
}


def many_buckets(seed, nb=300):
    r = np.random.default_rng(seed)
    ns = [int(4 * r.integers(1, 5000)) for _ in range(nb - 1)] + [int(r.integers(1, 20000))]
    ks = [int(r.integers(0, n + 1)) if r.random() < 0.2 else max(1, n // 100) for n in ns]
    return ns, ks


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from gradient_compression_ef_gb300 import gc
    ctx = gc.Context(8_000_000)
    yield torch, gc, ctx
    ctx.close()


def make_inputs(ns, seed, ties=False):
    r = np.random.default_rng(seed)
    n = sum(ns)
    if ties:  # few distinct magnitudes: thresholds fall inside long runs of ties
        g = (r.integers(-3, 4, size=n) * 0.5).astype(np.float32)
        e = (r.integers(-1, 2, size=n) * 0.25).astype(np.float32)
    else:
        g = r.standard_normal(n).astype(np.float32)
        e = (0.2 * r.standard_normal(n)).astype(np.float32)
    return g, e


def starts(ns):
    return np.concatenate([[0], np.cumsum(ns)]).astype(np.int64)


def run_topk(env, ns, ks, g, e):
    torch, gc, ctx = env
    ctx.set_buckets(ns, ks)
    oi, _, _ = gc.bucket_offsets(ks)
    gd = dev_f32(torch, g)
    ed = dev_f32(torch, e) if e is not None else None
    idx = torch.full((max(oi[-1], 4),), -7, dtype=torch.int32, device="cuda")
    val = torch.full((max(oi[-1], 4),), -7.0, dtype=torch.float32, device="cuda")
    gc.ef_topk_buckets(ctx, gd, ed, idx, val)
    ctx.check()
    return oi, host(idx), host(val), (host(ed) if ed is not None else None)


def check_topk(ns, ks, g, e, oi, idx, val, err, what):
    st = starts(ns)
    for b, (n, k) in enumerate(zip(ns, ks)):
        sl = slice(st[b], st[b + 1])
        o_idx, o_val, o_err = oracle.ef_topk(g[sl], None if e is None else e[sl], k)
        assert_bits_equal(idx[oi[b]:oi[b] + k], o_idx, "%s bucket %d idx" % (what, b))
        assert_bits_equal(val[oi[b]:oi[b] + k], o_val, "%s bucket %d val" % (what, b))
        if e is not None:
            assert_bits_equal(err[sl], o_err, "%s bucket %d err" % (what, b))


@pytest.mark.parametrize("name", sorted(LAYOUTS))
@pytest.mark.parametrize("ef", [True, False])
def test_topk_layouts(env, name, ef):
    ns, ks = LAYOUTS[name]
    g, e = make_inputs(ns, len(name))
    e = e if ef else None
    oi, idx, val, err = run_topk(env, ns, ks, g, e)
    check_topk(ns, ks, g, e, oi, idx, val, err, name)


@pytest.mark.parametrize("seed", [1, 2])
def test_topk_many_buckets(env, seed):
    ns, ks = many_buckets(seed)
    g, e = make_inputs(ns, seed)
    oi, idx, val, err = run_topk(env, ns, ks, g, e)
    check_topk(ns, ks, g, e, oi, idx, val, err, "many%d" % seed)


@pytest.mark.parametrize("name", ["segments", "mixed"])
def test_topk_heavy_ties(env, name):
    ns, ks = LAYOUTS[name]
    g, e = make_inputs(ns, 5, ties=True)
    oi, idx, val, err = run_topk(env, ns, ks, g, e)
    check_topk(ns, ks, g, e, oi, idx, val, err, name + " ties")


def test_topk_ties_beyond_the_stash(env):
    """Tens of thousands of entries share the threshold's top 23 key bits, more
    than the per-bucket stash holds: the refinement rescans the lists."""
    ns, ks = [120_000, 40_000], [7_000, 39_999]
    g = np.full(sum(ns), 1.5, np.float32)
    g[::7] = -1.5
    g[5::11] = np.float32(1.5) + np.float32(2.0 ** -22)   # a few just above
    e = np.zeros_like(g)
    oi, idx, val, err = run_topk(env, ns, ks, g, e)
    check_topk(ns, ks, g, e, oi, idx, val, err, "stash overflow")


def run_quant(env, ns, ks, g, e, bits, group, rounding, seed, step):
    torch, gc, ctx = env
    ctx.set_buckets(ns, ks)
    oi, oc, os_ = gc.bucket_offsets(ks, bits, group)
    gd, ed = dev_f32(torch, g), dev_f32(torch, e)
    idx = torch.full((max(oi[-1], 4),), -7, dtype=torch.int32, device="cuda")
    codes = torch.full((max(oc[-1], 16),), 0x5A, dtype=torch.uint8, device="cuda")
    scales = torch.full((max(os_[-1], 4),), -1.0, dtype=torch.float32, device="cuda")
    gc.ef_topk_quant_buckets(ctx, gd, ed, bits, group, rounding, seed, step, idx, codes, scales)
    ctx.check()
    return (oi, oc, os_), host(idx), host(codes), host(scales), host(ed)


def check_quant(ns, ks, g, e, bits, group, rounding, seed, step, offs, idx, codes, scales, err,
                what):
    oi, oc, os_ = offs
    st = starts(ns)
    for b, (n, k) in enumerate(zip(ns, ks)):
        sl = slice(st[b], st[b + 1])
        o_idx, o_codes, o_scales, o_err = oracle.ef_topk_quant(
            g[sl], e[sl], k, bits, group, rounding, oracle.bucket_seed(seed, b), step)
        w = "%s bucket %d" % (what, b)
        assert_bits_equal(idx[oi[b]:oi[b] + k], o_idx, w + " idx")
        assert o_codes.size == oc[b + 1] - oc[b]
        assert_bits_equal(codes[oc[b]:oc[b + 1]], o_codes, w + " codes")
        assert_bits_equal(scales[os_[b]:os_[b] + o_scales.size], o_scales, w + " scales")
        assert_bits_equal(err[sl], o_err, w + " err")


@pytest.mark.parametrize("name", ["tiny", "segments", "mixed", "single"])
@pytest.mark.parametrize("bits", [8, 4, 2, 1])
@pytest.mark.parametrize("rounding", ["nearest_even", "stochastic"])
def test_quant_layouts(env, name, bits, rounding):
    ns, ks = LAYOUTS[name]
    g, e = make_inputs(ns, bits)
    out = run_quant(env, ns, ks, g, e, bits, 64, rounding, 11, 3)
    check_quant(ns, ks, g, e, bits, 64, rounding, 11, 3, *out, name)


@pytest.mark.parametrize("group", [4, 8, 32, 128])
def test_quant_groups(env, group):
    ns, ks = LAYOUTS["mixed"]
    g, e = make_inputs(ns, group)
    out = run_quant(env, ns, ks, g, e, 8, group, "stochastic", 5, 1)
    check_quant(ns, ks, g, e, 8, group, "stochastic", 5, 1, *out, "g%d" % group)


def test_quant_many_buckets(env):
    ns, ks = many_buckets(9, nb=120)
    g, e = make_inputs(ns, 9)
    out = run_quant(env, ns, ks, g, e, 4, 16, "stochastic", 100, 7)
    check_quant(ns, ks, g, e, 4, 16, "stochastic", 100, 7, *out, "many")


def test_error_feedback_steps_match_single_calls(env):
    """Several correlated EF steps: the bucketed call and the per-bucket
    calls keep identical residuals and outputs step after step (the plan's
    state is reset by every call)."""
    torch, gc, ctx = env
    ns, ks = [262_144, 131_072, 65_540, 30_001], [2_621, 1_310, 655, 300]
    n = sum(ns)
    st = starts(ns)
    ctx.set_buckets(ns, ks)
    oi, oc, os_ = gc.bucket_offsets(ks, 8, 64)
    grads = inputs.correlated_steps(n, 4, seed=3)
    e_bk = torch.zeros(n, dtype=torch.float32, device="cuda")
    e_one = torch.zeros(n, dtype=torch.float32, device="cuda")
    idx_bk = torch.empty(oi[-1], dtype=torch.int32, device="cuda")
    codes_bk = torch.empty(oc[-1], dtype=torch.uint8, device="cuda")
    scales_bk = torch.empty(os_[-1], dtype=torch.float32, device="cuda")
    idx_one, codes_one, scales_one = (torch.empty_like(idx_bk), torch.empty_like(codes_bk),
                                      torch.empty_like(scales_bk))
    for step, g in enumerate(grads):
        gd = dev_f32(torch, g)
        gc.ef_topk_quant_buckets(ctx, gd, e_bk, 8, 64, "stochastic", 50, step, idx_bk,
                                 codes_bk, scales_bk)
        for b, (nb_, kb) in enumerate(zip(ns, ks)):
            s0 = int(st[b])
            gc.ef_topk_quant(ctx, gd[s0:s0 + nb_], e_one[s0:s0 + nb_], kb, 8, 64, "stochastic",
                             gc.bucket_seed(50, b), step, idx_one[oi[b]:oi[b] + kb],
                             codes_one[oc[b]:oc[b + 1]], scales_one[os_[b]:os_[b + 1]])
        ctx.check()
        assert_bits_equal(host(e_bk), host(e_one), "step %d err" % step)
        for b, kb in enumerate(ks):
            assert_bits_equal(host(idx_bk)[oi[b]:oi[b] + kb], host(idx_one)[oi[b]:oi[b] + kb],
                              "step %d idx %d" % (step, b))
        assert_bits_equal(host(codes_bk), host(codes_one), "step %d codes" % step)
        nsc = [gc.scales_floats(kb, 64, "qsgd") for kb in ks]
        for b in range(len(ks)):
            assert_bits_equal(host(scales_bk)[os_[b]:os_[b] + nsc[b]],
                              host(scales_one)[os_[b]:os_[b] + nsc[b]], "step %d scales" % step)


def test_launches_per_call_do_not_grow_with_buckets(env):
    torch, gc, ctx = env
    for ns, ks in (LAYOUTS["tiny"], many_buckets(4, nb=200)):
        ctx.set_buckets(ns, ks)
        oi, oc, os_ = gc.bucket_offsets(ks, 8, 64)
        n = sum(ns)
        gd = torch.randn(n, device="cuda")
        ed = torch.zeros(n, device="cuda")
        idx = torch.empty(max(oi[-1], 4), dtype=torch.int32, device="cuda")
        codes = torch.empty(max(oc[-1], 16), dtype=torch.uint8, device="cuda")
        scales = torch.empty(max(os_[-1], 4), dtype=torch.float32, device="cuda")
        before = ctx.launch_count()
        gc.ef_topk_quant_buckets(ctx, gd, ed, 8, 64, "nearest_even", 0, 0, idx, codes, scales)
        assert ctx.launch_count() - before == 5
        val = torch.empty(max(oi[-1], 4), dtype=torch.float32, device="cuda")
        before = ctx.launch_count()
        gc.ef_topk_buckets(ctx, gd, ed, idx, val)
        assert ctx.launch_count() - before == 4
        ctx.check()


def test_graph_replay_matches_eager(env):
    torch, gc, ctx = env
    ns, ks = LAYOUTS["mixed"]
    g, e = make_inputs(ns, 21)
    ctx.set_buckets(ns, ks)
    oi, oc, os_ = gc.bucket_offsets(ks, 8, 64)
    gd = dev_f32(torch, g)
    outs = []
    for mode in ("eager", "graph"):
        ed = dev_f32(torch, e)
        idx = torch.zeros(oi[-1], dtype=torch.int32, device="cuda")
        codes = torch.zeros(oc[-1], dtype=torch.uint8, device="cuda")
        scales = torch.zeros(os_[-1], dtype=torch.float32, device="cuda")
        if mode == "eager":
            for step in range(2):
                gc.ef_topk_quant_buckets(ctx, gd, ed, 8, 64, "stochastic", 1, 0, idx, codes,
                                         scales)
        else:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            ctx.set_stream(s)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s):
                gc.ef_topk_quant_buckets(ctx, gd, ed, 8, 64, "stochastic", 1, 0, idx, codes,
                                         scales)
            torch.cuda.current_stream().wait_stream(s)
            ctx.set_stream(torch.cuda.current_stream())
            ed.copy_(dev_f32(torch, e))
            graph.replay()
            graph.replay()
            torch.cuda.synchronize()
        ctx.check()
        outs.append((host(ed), host(idx), host(codes), host(scales)))
    for a, b, what in zip(outs[0], outs[1], ("err", "idx", "codes", "scales")):
        assert_bits_equal(b, a, "graph " + what)


def test_plan_and_call_validation(env):
    torch, gc, ctx = env
    fresh = gc.Context(0)
    x = torch.zeros(64, device="cuda")
    i = torch.zeros(64, dtype=torch.int32, device="cuda")
    with pytest.raises(gc.GCError) as ex:
        gc.ef_topk_buckets(fresh, x, x, i, x)
    assert ex.value.status == gc.ERR_WORKSPACE
    for ns, ks, status in (([6, 8], [1, 1], gc.ERR_ALIGNMENT), ([8, 8], [9, 1], gc.ERR_INVALID_ARG),
                           ([8, 0], [1, 0], gc.ERR_INVALID_ARG), ([], [], gc.ERR_INVALID_ARG)):
        with pytest.raises(gc.GCError) as ex:
            fresh.set_buckets(ns, ks)
        assert ex.value.status == status, (ns, ks)
    fresh.set_buckets([32, 32], [4, 4])
    c = torch.zeros(64, dtype=torch.uint8, device="cuda")
    for group in (0, 2, 48, 256):
        with pytest.raises(gc.GCError) as ex:
            gc.ef_topk_quant_buckets(fresh, x, x, 8, group, "stochastic", 0, 0, i, c, x)
        assert ex.value.status == gc.ERR_UNSUPPORTED
    with pytest.raises(gc.GCError) as ex:
        gc.ef_topk_quant_buckets(fresh, x, None, 8, 64, "stochastic", 0, 0, i, c, x)
    assert ex.value.status == gc.ERR_INVALID_ARG
    with pytest.raises(gc.GCError) as ex:
        gc.ef_topk_buckets(fresh, x[1:], x, i, x)
    assert ex.value.status == gc.ERR_ALIGNMENT
    fresh.close()


def test_full_size_workload(env):
    """The 134,217,728-element gradient in 21 buckets of 25 MiB, Top-K 1 % +
    8-bit QSGD (groups of 64, stochastic), two correlated EF steps: every
    bucket equals the single-bucket call bit for bit, and the first and last
    buckets equal the oracle."""
    torch, gc, _ = env
    n = inputs.FLAT_ELEMS
    bounds = inputs.bucket_bounds(n)
    ns = [length for _, length in bounds]
    ks = [inputs.ratio_k(length, 10, 1000) for length in ns]
    ctx = gc.Context(max(ns))
    ctx.set_buckets(ns, ks)
    oi, oc, os_ = gc.bucket_offsets(ks, 8, 64)
    grads = inputs.correlated_steps_device(n, 2, "cuda", seed=5)
    e_bk = torch.zeros(n, dtype=torch.float32, device="cuda")
    e_one = torch.zeros(n, dtype=torch.float32, device="cuda")
    out_bk = [torch.empty(oi[-1], dtype=torch.int32, device="cuda"),
              torch.empty(oc[-1], dtype=torch.uint8, device="cuda"),
              torch.empty(os_[-1], dtype=torch.float32, device="cuda")]
    out_one = [torch.empty_like(t) for t in out_bk]
    e_before = None
    for step, gd in enumerate(grads):
        if step == len(grads) - 1:
            e_before = host(e_bk)
        gc.ef_topk_quant_buckets(ctx, gd, e_bk, 8, 64, "stochastic", 1000, step, *out_bk)
        for b, ((s0, length), kb) in enumerate(zip(bounds, ks)):
            gc.ef_topk_quant(ctx, gd[s0:s0 + length], e_one[s0:s0 + length], kb, 8, 64,
                             "stochastic", gc.bucket_seed(1000, b), step,
                             out_one[0][oi[b]:oi[b] + kb],
                             out_one[1][oc[b]:oc[b + 1]], out_one[2][os_[b]:os_[b + 1]])
        ctx.check()
    assert_bits_equal(host(e_bk), host(e_one), "full err")
    assert_bits_equal(host(out_bk[1]), host(out_one[1]), "full codes")
    i_bk, i_one, s_bk, s_one = (host(t) for t in (out_bk[0], out_one[0], out_bk[2], out_one[2]))
    for b, kb in enumerate(ks):
        assert_bits_equal(i_bk[oi[b]:oi[b] + kb], i_one[oi[b]:oi[b] + kb], "full idx %d" % b)
        ns_ = gc.scales_floats(kb, 64, "qsgd")
        assert_bits_equal(s_bk[os_[b]:os_[b] + ns_], s_one[os_[b]:os_[b] + ns_],
                          "full scales %d" % b)
    g_last = host(grads[-1])
    idx_h, codes_h, scales_h, err_h = (host(t) for t in (*out_bk, e_bk))
    for b in (0, len(bounds) - 1):
        s0, length = bounds[b]
        sl = slice(s0, s0 + length)
        o_idx, o_codes, o_scales, o_err = oracle.ef_topk_quant(
            g_last[sl], e_before[sl], ks[b], 8, 64, "stochastic", oracle.bucket_seed(1000, b),
            len(grads) - 1)
        assert_bits_equal(idx_h[oi[b]:oi[b] + ks[b]], o_idx, "oracle idx %d" % b)
        assert_bits_equal(codes_h[oc[b]:oc[b + 1]], o_codes, "oracle codes %d" % b)
        assert_bits_equal(scales_h[os_[b]:os_[b] + o_scales.size], o_scales, "oracle scales %d" % b)
        assert_bits_equal(err_h[sl], o_err, "oracle err %d" % b)
    ctx.close()


@pytest.mark.parametrize("scales", [(1.0, 1.0, 0.25, 4.0, 1.0), (1.0, 0.97, 1.03, 16.0, 0.01)])
def test_threshold_guess_paths(env, scales):
    """The hist pass lists entries from a little below the previous call's
    threshold bin.  Calls whose magnitudes drop (the guess is too high: the
    collect pass reads c again) or rise (long lists) give exactly the
    oracle's result, as do steady calls that use the lists alone."""
    torch, gc, ctx = env
    ns, ks = [65_536, 131_072, 40_000], [655, 1_310, 400]
    ctx.set_buckets(ns, ks)
    oi, oc, os_ = gc.bucket_offsets(ks, 8, 64)
    st = starts(ns)
    r = np.random.default_rng(17)
    base = inputs.student_t(r, sum(ns))
    e = np.zeros(sum(ns), np.float32)
    ed = dev_f32(torch, e)
    idx = torch.empty(oi[-1], dtype=torch.int32, device="cuda")
    codes = torch.empty(oc[-1], dtype=torch.uint8, device="cuda")
    scl = torch.empty(os_[-1], dtype=torch.float32, device="cuda")
    for step, f in enumerate(scales):
        g = (base * np.float32(f)).astype(np.float32)
        gc.ef_topk_quant_buckets(ctx, dev_f32(torch, g), ed, 8, 64, "stochastic", 3, step, idx,
                                 codes, scl)
        ctx.check()
        e_new, i_h, c_h, s_h = host(ed), host(idx), host(codes), host(scl)
        for b, (n, k) in enumerate(zip(ns, ks)):
            sl = slice(st[b], st[b + 1])
            o_idx, o_codes, o_scales, o_err = oracle.ef_topk_quant(
                g[sl], e[sl], k, 8, 64, "stochastic", oracle.bucket_seed(3, b), step)
            w = "step %d bucket %d" % (step, b)
            assert_bits_equal(i_h[oi[b]:oi[b] + k], o_idx, w + " idx")
            assert_bits_equal(c_h[oc[b]:oc[b + 1]], o_codes, w + " codes")
            assert_bits_equal(s_h[os_[b]:os_[b] + o_scales.size], o_scales, w + " scales")
            assert_bits_equal(e_new[sl], o_err, w + " err")
        e = e_new
