"""Deferred residual write-back of the bucketed hybrid on the GPU.

With the context's deferred mode on, a call leaves e' = c at its kept
positions and the next call on the same error buffer applies the kept
entries' residuals while it reads e.  Every output (indices, codes, scales,
diagnostics) must equal the immediate write-back bit for bit, step after
step, and so must the error buffer once flushed; the immediate path is the
one pinned to the oracle, and one chain here goes to the oracle directly."""
import numpy as np
import pytest

import oracle
from gradient_compression_ef_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, dev_f32, host, torch_cuda
from tests.test_gpu_buckets import LAYOUTS, make_inputs, many_buckets, starts

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from gradient_compression_ef_gb300 import gc
    now = gc.Context(0)
    later = gc.Context(0)
    later.set_deferred_residual(True)
    yield torch, gc, now, later
    now.close()
    later.close()


class Outs:
    """Output buffers of one context for a plan."""

    def __init__(self, torch, gc, ks, bits, group, diag):
        oi, oc, os_ = gc.bucket_offsets(ks, bits, group)
        self.offs = (oi, oc, os_)
        self.idx = torch.full((max(oi[-1], 4),), -7, dtype=torch.int32, device="cuda")
        self.codes = torch.full((max(oc[-1], 16),), 0x5A, dtype=torch.uint8, device="cuda")
        self.scales = torch.full((max(os_[-1], 4),), -1.0, dtype=torch.float32, device="cuda")
        self.diag = (torch.zeros(3 * len(ks), dtype=torch.float64, device="cuda")
                     if diag else None)

    def snapshot(self):
        d = host(self.diag) if self.diag is not None else None
        return host(self.idx), host(self.codes), host(self.scales), d


def compare(a, b, ks, offs, what):
    oi = offs[0]
    for b_, k in enumerate(ks):
        assert_bits_equal(b[0][oi[b_]:oi[b_] + k], a[0][oi[b_]:oi[b_] + k],
                          "%s bucket %d idx" % (what, b_))
    assert_bits_equal(b[1], a[1], what + " codes")
    assert_bits_equal(b[2], a[2], what + " scales")
    if a[3] is not None:
        assert np.array_equal(a[3].view(np.uint64), b[3].view(np.uint64)), what + " diag"


def run_pair(env, ns, ks, grads, e0, bits=8, group=64, rounding="stochastic", seed=31,
             diag=False, flush_at=()):
    """Steps through grads on both contexts; returns the immediate context's
    final err and the deferred one's after a flush."""
    torch, gc, now, later = env
    now.set_buckets(ns, ks)
    later.set_buckets(ns, ks)
    on, ol = (Outs(torch, gc, ks, bits, group, diag) for _ in range(2))
    e_now, e_later = dev_f32(torch, e0), dev_f32(torch, e0)
    for step, g in enumerate(grads):
        gd = dev_f32(torch, g)
        gc.ef_topk_quant_buckets(now, gd, e_now, bits, group, rounding, seed, step, on.idx,
                                 on.codes, on.scales, diag=on.diag)
        gc.ef_topk_quant_buckets(later, gd, e_later, bits, group, rounding, seed, step, ol.idx,
                                 ol.codes, ol.scales, diag=ol.diag)
        now.check()
        later.check()
        compare(on.snapshot(), ol.snapshot(), ks, on.offs, "step %d" % step)
        if step in flush_at:
            later.bucket_flush()
            assert_bits_equal(host(e_later), host(e_now), "step %d flushed err" % step)
    later.bucket_flush()
    later.check()
    return host(e_now), host(e_later)


@pytest.mark.parametrize("name", ["tiny", "segments", "mixed", "single", "one_element"])
@pytest.mark.parametrize("diag", [False, True])
def test_deferred_steps_match_immediate(env, name, diag):
    ns, ks = LAYOUTS[name]
    n = sum(ns)
    grads = list(inputs.correlated_steps(n, 4, seed=len(name)))
    _, e0 = make_inputs(ns, 3)
    a, b = run_pair(env, ns, ks, grads, e0, diag=diag, flush_at=(1,))
    assert_bits_equal(b, a, name + " err")


@pytest.mark.parametrize("bits,group,rounding", [(4, 16, "nearest_even"), (2, 128, "stochastic"),
                                                 (1, 4, "stochastic")])
def test_deferred_bits_and_groups(env, bits, group, rounding):
    ns, ks = LAYOUTS["segments"]
    grads = list(inputs.correlated_steps(sum(ns), 3, seed=bits))
    _, e0 = make_inputs(ns, bits)
    a, b = run_pair(env, ns, ks, grads, e0, bits, group, rounding)
    assert_bits_equal(b, a, "b%d g%d err" % (bits, group))


def test_deferred_many_buckets_and_dense_segments(env):
    """Buckets with k up to n: segments with hundreds to 2048 kept entries
    walk the 64-entry window many times inside one pass."""
    ns, ks = many_buckets(17, nb=150)
    grads = list(inputs.correlated_steps(sum(ns), 3, seed=17))
    _, e0 = make_inputs(ns, 17)
    a, b = run_pair(env, ns, ks, grads, e0, 8, 32, "stochastic", diag=True)
    assert_bits_equal(b, a, "many err")


def test_deferred_ties(env):
    """Few distinct magnitudes: the kept ties of a segment end its run of
    entries; their residuals land exactly once."""
    ns, ks = LAYOUTS["segments"]
    g0, e0 = make_inputs(ns, 5, ties=True)
    g1, _ = make_inputs(ns, 6, ties=True)
    a, b = run_pair(env, ns, ks, [g0, g1, g0, g1], e0)
    assert_bits_equal(b, a, "ties err")


def test_deferred_chain_against_oracle(env):
    """Three deferred steps and a flush against the oracle's chain of
    immediate steps, bucket by bucket."""
    torch, gc, _, later = env
    ns, ks = LAYOUTS["segments"]
    st = starts(ns)
    grads = list(inputs.correlated_steps(sum(ns), 3, seed=8))
    _, e0 = make_inputs(ns, 8)
    later.set_buckets(ns, ks)
    ol = Outs(torch, gc, ks, 8, 64, False)
    ed = dev_f32(torch, e0)
    e_or = [e0[st[b]:st[b + 1]].copy() for b in range(len(ns))]
    for step, g in enumerate(grads):
        gc.ef_topk_quant_buckets(later, dev_f32(torch, g), ed, 8, 64, "stochastic", 40, step,
                                 ol.idx, ol.codes, ol.scales)
        idx, codes, scales, _ = ol.snapshot()
        oi, oc, os_ = ol.offs
        for b, k in enumerate(ks):
            o_idx, o_codes, o_scales, e_or[b] = oracle.ef_topk_quant(
                g[st[b]:st[b + 1]], e_or[b], k, 8, 64, "stochastic", oracle.bucket_seed(40, b),
                step)
            assert_bits_equal(idx[oi[b]:oi[b] + k], o_idx, "step %d bucket %d idx" % (step, b))
            assert_bits_equal(codes[oc[b]:oc[b + 1]], o_codes, "step %d codes" % step)
            assert_bits_equal(scales[os_[b]:os_[b] + o_scales.size], o_scales,
                              "step %d scales" % step)
    later.bucket_flush()
    later.check()
    assert_bits_equal(host(ed), np.concatenate(e_or), "flushed err")


def test_deferred_graph_replay(env):
    """A deferred call captured into a CUDA graph applies at each replay the
    residuals the previous replay left."""
    torch, gc, now, later = env
    ns, ks = LAYOUTS["mixed"]
    g, e0 = make_inputs(ns, 12)
    gd = dev_f32(torch, g)
    now.set_buckets(ns, ks)
    later.set_buckets(ns, ks)
    on, ol = Outs(torch, gc, ks, 8, 64, False), Outs(torch, gc, ks, 8, 64, False)
    e_now, e_later = dev_f32(torch, e0), dev_f32(torch, e0)
    for _ in range(4):
        gc.ef_topk_quant_buckets(now, gd, e_now, 8, 64, "stochastic", 2, 0, on.idx, on.codes,
                                 on.scales)
    gc.ef_topk_quant_buckets(later, gd, e_later, 8, 64, "stochastic", 2, 0, ol.idx, ol.codes,
                             ol.scales)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    later.set_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        gc.ef_topk_quant_buckets(later, gd, e_later, 8, 64, "stochastic", 2, 0, ol.idx,
                                 ol.codes, ol.scales)
    # replays run on the current stream: the flush goes there after them
    torch.cuda.current_stream().wait_stream(s)
    later.set_stream(torch.cuda.current_stream())
    for _ in range(3):
        graph.replay()
    later.bucket_flush()
    torch.cuda.synchronize()
    later.check()
    now.check()
    compare(on.snapshot(), ol.snapshot(), ks, on.offs, "graph")
    assert_bits_equal(host(e_later), host(e_now), "graph err")


def test_deferred_rules(env):
    torch, gc, now, later = env
    ns, ks = LAYOUTS["mixed"]
    n = sum(ns)
    g, e0 = make_inputs(ns, 14)
    gd = dev_f32(torch, g)
    later.set_buckets(ns, ks)
    now.set_buckets(ns, ks)
    o = Outs(torch, gc, ks, 8, 64, False)
    e_now = dev_f32(torch, e0)
    for _ in range(2):
        gc.ef_topk_quant_buckets(now, gd, e_now, 8, 64, "nearest_even", 0, 0, o.idx, o.codes,
                                 o.scales)
    ed, other = dev_f32(torch, e0), dev_f32(torch, e0)
    later.bucket_flush()  # nothing pending: no launch
    before = later.launch_count()
    later.bucket_flush()
    assert later.launch_count() == before
    gc.ef_topk_quant_buckets(later, gd, ed, 8, 64, "nearest_even", 0, 0, o.idx, o.codes, o.scales)
    assert later.launch_count() - before == 5
    # pending residuals belong to ed: a call on another buffer, or on none, is refused
    with pytest.raises(gc.GCError) as ex:
        gc.ef_topk_quant_buckets(later, gd, other, 8, 64, "nearest_even", 0, 0, o.idx, o.codes,
                                 o.scales)
    assert ex.value.status == gc.ERR_INVALID_ARG
    val = torch.empty(o.idx.numel(), dtype=torch.float32, device="cuda")
    for e_arg in (other, None):
        with pytest.raises(gc.GCError) as ex:
            gc.ef_topk_buckets(later, gd, e_arg, o.idx, val)
        assert ex.value.status == gc.ERR_INVALID_ARG
    assert later.launch_count() - before == 5
    # the second call applies the first one's residuals
    gc.ef_topk_quant_buckets(later, gd, ed, 8, 64, "nearest_even", 0, 0, o.idx, o.codes, o.scales)
    # switching the mode off flushes
    later.set_deferred_residual(False)
    assert later.launch_count() - before == 11
    later.check()
    assert_bits_equal(host(ed), host(e_now), "flushed by mode off")
    gc.ef_topk_buckets(later, gd, other, o.idx, val)  # allowed again
    later.set_deferred_residual(True)
    # re-planning flushes first
    ed2 = dev_f32(torch, e0)
    gc.ef_topk_quant_buckets(later, gd, ed2, 8, 64, "nearest_even", 0, 0, o.idx, o.codes,
                             o.scales)
    gc.ef_topk_quant_buckets(later, gd, ed2, 8, 64, "nearest_even", 0, 0, o.idx, o.codes,
                             o.scales)
    later.set_buckets(ns, ks)
    later.check()
    assert_bits_equal(host(ed2), host(e_now), "flushed by re-planning")
    assert n == ed2.numel()


def test_deferred_full_size_workload(env):
    """The 134,217,728-element gradient in 21 buckets of 25 MiB, Top-K 1 % +
    8-bit QSGD: three correlated steps deferred equal the immediate ones."""
    torch, gc, now, later = env
    bounds = inputs.bucket_bounds(inputs.FLAT_ELEMS)
    ns = [l for _, l in bounds]
    ks = [inputs.ratio_k(l, 1, 100) for l in ns]
    now.set_buckets(ns, ks)
    later.set_buckets(ns, ks)
    grads = inputs.correlated_steps_device(inputs.FLAT_ELEMS, 3, "cuda", seed=5)
    on, ol = Outs(torch, gc, ks, 8, 64, True), Outs(torch, gc, ks, 8, 64, True)
    e_now = torch.zeros(inputs.FLAT_ELEMS, dtype=torch.float32, device="cuda")
    e_later = torch.zeros_like(e_now)
    for step, gd in enumerate(grads):
        gc.ef_topk_quant_buckets(now, gd, e_now, 8, 64, "stochastic", 1000, step, on.idx,
                                 on.codes, on.scales, diag=on.diag)
        gc.ef_topk_quant_buckets(later, gd, e_later, 8, 64, "stochastic", 1000, step, ol.idx,
                                 ol.codes, ol.scales, diag=ol.diag)
        compare(on.snapshot(), ol.snapshot(), ks, on.offs, "full step %d" % step)
    later.bucket_flush()
    now.check()
    later.check()
    assert torch.equal(e_now.view(torch.int32), e_later.view(torch.int32))


def test_deferred_graph_captured_first(env):
    """A deferred call captured before any call of the plan ran: the first
    replay finds nothing pending, every later one applies the residuals of
    the replay before it; a flush after the replays completes e'."""
    torch, gc, now, later = env
    ns, ks = LAYOUTS["segments"]
    g, e0 = make_inputs(ns, 19)
    gd = dev_f32(torch, g)
    now.set_buckets(ns, ks)
    later.set_buckets(ns, ks)
    on, ol = Outs(torch, gc, ks, 8, 64, False), Outs(torch, gc, ks, 8, 64, False)
    e_now, e_later = dev_f32(torch, e0), dev_f32(torch, e0)
    for _ in range(4):
        gc.ef_topk_quant_buckets(now, gd, e_now, 8, 64, "stochastic", 6, 2, on.idx, on.codes,
                                 on.scales)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    later.set_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        gc.ef_topk_quant_buckets(later, gd, e_later, 8, 64, "stochastic", 6, 2, ol.idx,
                                 ol.codes, ol.scales)
    torch.cuda.current_stream().wait_stream(s)
    later.set_stream(torch.cuda.current_stream())
    for _ in range(4):
        graph.replay()
    later.bucket_flush()
    torch.cuda.synchronize()
    later.check()
    now.check()
    compare(on.snapshot(), ol.snapshot(), ks, on.offs, "captured first")
    assert_bits_equal(host(e_later), host(e_now), "captured first err")


def test_deferred_flush_then_new_error_buffer_contents(env):
    """After a flush the plan holds nothing pending: new contents written into
    e (a checkpoint restored, say) are not overwritten by old residuals."""
    torch, gc, now, later = env
    ns, ks = LAYOUTS["mixed"]
    g, e0 = make_inputs(ns, 23)
    _, e1 = make_inputs(ns, 24)
    gd = dev_f32(torch, g)
    now.set_buckets(ns, ks)
    later.set_buckets(ns, ks)
    on, ol = Outs(torch, gc, ks, 8, 64, False), Outs(torch, gc, ks, 8, 64, False)
    ed = dev_f32(torch, e0)
    for step in range(2):
        gc.ef_topk_quant_buckets(later, gd, ed, 8, 64, "stochastic", 3, step, ol.idx, ol.codes,
                                 ol.scales)
    later.bucket_flush()
    ed.copy_(dev_f32(torch, e1))
    e_now = dev_f32(torch, e1)
    for step in range(2, 4):
        gc.ef_topk_quant_buckets(now, gd, e_now, 8, 64, "stochastic", 3, step, on.idx, on.codes,
                                 on.scales)
        gc.ef_topk_quant_buckets(later, gd, ed, 8, 64, "stochastic", 3, step, ol.idx, ol.codes,
                                 ol.scales)
        compare(on.snapshot(), ol.snapshot(), ks, on.offs, "restored step %d" % step)
    later.bucket_flush()
    torch.cuda.synchronize()
    later.check()
    now.check()
    assert_bits_equal(host(ed), host(e_now), "restored err")


def run_topk_pair(env, ns, ks, grads, e0, calls, diag=False):
    """Top-K-only (and, where calls says so, hybrid) bucketed steps on both
    contexts; compares every output and the flushed err."""
    torch, gc, now, later = env
    now.set_buckets(ns, ks)
    later.set_buckets(ns, ks)
    oi, _, _ = gc.bucket_offsets(ks)
    on, ol = Outs(torch, gc, ks, 8, 64, diag), Outs(torch, gc, ks, 8, 64, diag)
    vals = [torch.full((max(oi[-1], 4),), -7.0, dtype=torch.float32, device="cuda")
            for _ in range(2)]
    e_now, e_later = dev_f32(torch, e0), dev_f32(torch, e0)
    for step, (g, kind) in enumerate(zip(grads, calls)):
        gd = dev_f32(torch, g)
        for ctx, o, v, e in ((now, on, vals[0], e_now), (later, ol, vals[1], e_later)):
            if kind == "topk":
                gc.ef_topk_buckets(ctx, gd, e, o.idx, v, diag=o.diag)
            else:
                gc.ef_topk_quant_buckets(ctx, gd, e, 8, 64, "stochastic", 9, step, o.idx,
                                         o.codes, o.scales, diag=o.diag)
        now.check()
        later.check()
        a, b = on.snapshot(), ol.snapshot()
        for b_, k in enumerate(ks):
            assert_bits_equal(b[0][oi[b_]:oi[b_] + k], a[0][oi[b_]:oi[b_] + k],
                              "step %d bucket %d idx" % (step, b_))
            if kind == "topk":
                assert_bits_equal(host(vals[1])[oi[b_]:oi[b_] + k],
                                  host(vals[0])[oi[b_]:oi[b_] + k], "step %d val" % step)
        if kind != "topk":
            compare(a, b, ks, on.offs, "step %d" % step)
        elif diag:
            assert np.array_equal(a[3].view(np.uint64), b[3].view(np.uint64)), "diag"
    later.bucket_flush()
    later.check()
    assert_bits_equal(host(e_later), host(e_now), "flushed err")


@pytest.mark.parametrize("name", ["tiny", "segments", "mixed", "one_element"])
@pytest.mark.parametrize("diag", [False, True])
def test_deferred_topk_steps_match_immediate(env, name, diag):
    """Top-K only: the kept entries' e' = +0 is deferred the same way."""
    ns, ks = LAYOUTS[name]
    grads = list(inputs.correlated_steps(sum(ns), 4, seed=30 + len(name)))
    _, e0 = make_inputs(ns, 31)
    run_topk_pair(env, ns, ks, grads, e0, ["topk"] * 4, diag)


def test_deferred_topk_and_hybrid_interleaved(env):
    """Top-K and hybrid steps on one error buffer: each applies what the call
    before it left, whichever kind that was."""
    ns, ks = many_buckets(33, nb=60)
    grads = list(inputs.correlated_steps(sum(ns), 5, seed=33))
    _, e0 = make_inputs(ns, 33)
    run_topk_pair(env, ns, ks, grads, e0, ["topk", "quant", "quant", "topk", "quant"])
