"""gc_ef_topk_noalloc -- the allocation-free EF + Top-K entry point.

Some callers cannot allocate device memory (their memory belongs to another
allocator, or they run under a hard budget or on a path where cudaMalloc's
device-wide synchronisation is not acceptable), so they cannot create a
context.  This entry point keeps its scratch in a static device array of the
library instead.  Here it is called through the C ABI and must give exactly
what gc_ef_topk with a context gives on the same inputs: over two calls in a
row (two error-feedback steps), over the edge cases of k and of the error
buffer, at its maximum size, and for a small call right after a large one
(each call clears only the leading part of the shared array).  A last test
checks the property that names it: repeated calls leave the device's free
memory and torch's allocator unchanged.

No test here depends on running after the others.  The file's name sorts
last so that pytest collects it last: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest

from tests.gpu_helpers import assert_bits_equal, dev_f32, host, torch_cuda

pytestmark = pytest.mark.gpu


def _outputs(torch, k):
    k = max(k, 1)
    return (torch.full((k,), -1, dtype=torch.int32, device="cuda"),
            torch.full((k,), -1.0, dtype=torch.float32, device="cuda"))


def _noalloc(gc, torch, gd, ed, n, k, idx, val):
    st = gc.lib.gc_ef_topk_noalloc(gd.data_ptr(), ed.data_ptr() if ed is not None else None,
                                   n, k, idx.data_ptr(), val.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert st == gc.OK, gc.status_string(st)


def _compare(torch, gc, ctx, g, e0, k, what):
    """One call of each entry point on the same inputs; every output and
    the residual bit for bit."""
    n = g.size
    gd = dev_f32(torch, g)
    e_ctx = dev_f32(torch, e0) if e0 is not None else None
    e_na = dev_f32(torch, e0) if e0 is not None else None
    i_ctx, v_ctx = _outputs(torch, k)
    gc.ef_topk(ctx, gd, e_ctx, k, i_ctx, v_ctx)
    ctx.check()
    i_na, v_na = _outputs(torch, k)
    _noalloc(gc, torch, gd, e_na, n, k, i_na, v_na)
    torch.cuda.synchronize()
    assert_bits_equal(host(i_na)[:k], host(i_ctx)[:k], what + " idx")
    assert_bits_equal(host(v_na)[:k], host(v_ctx)[:k], what + " val")
    if e0 is not None:
        assert_bits_equal(host(e_na), host(e_ctx), what + " err")


def test_noalloc_matches_context_call_on_two_calls_in_a_row():
    torch = torch_cuda()
    from gradient_compression_ef_gb300 import gc
    r = np.random.default_rng(20261202)
    n, k = 1_000_003, 10_000
    g1 = r.standard_normal(n).astype(np.float32)
    g2 = r.standard_normal(n).astype(np.float32)
    e0 = (0.1 * r.standard_normal(n)).astype(np.float32)

    e_ctx, e_na = dev_f32(torch, e0), dev_f32(torch, e0)
    with gc.Context(n) as ctx:
        for step, g in enumerate((g1, g2)):
            gd = dev_f32(torch, g)
            i_ctx, v_ctx = _outputs(torch, k)
            gc.ef_topk(ctx, gd, e_ctx, k, i_ctx, v_ctx)
            ctx.check()
            i_na, v_na = _outputs(torch, k)
            _noalloc(gc, torch, gd, e_na, n, k, i_na, v_na)
            torch.cuda.synchronize()
            what = "call %d" % (step + 1)
            assert_bits_equal(host(i_na), host(i_ctx), what + " idx")
            assert_bits_equal(host(v_na), host(v_ctx), what + " val")
            assert_bits_equal(host(e_na), host(e_ctx), what + " err")


MAX_N = 1048576  # GC_NOALLOC_MAX_N


@pytest.mark.parametrize("n,k", [(1, 1), (300, 7), (MAX_N, MAX_N // 100), (4097, 4097),
                                 (5000, 0)])
@pytest.mark.parametrize("with_err", [True, False])
def test_noalloc_edge_cases(n, k, with_err):
    torch = torch_cuda()
    from gradient_compression_ef_gb300 import gc
    assert gc.NOALLOC_MAX_N == MAX_N
    r = np.random.default_rng(n + k)
    g = r.standard_normal(n).astype(np.float32)
    e0 = (0.3 * r.standard_normal(n)).astype(np.float32) if with_err else None
    with gc.Context(n) as ctx:
        _compare(torch, gc, ctx, g, e0, k, "n=%d k=%d err=%s" % (n, k, with_err))


def test_noalloc_small_call_after_a_large_one():
    """A maximum-size call leaves counters, histograms and candidates in the
    shared array; the small call after it must not see any of them."""
    torch = torch_cuda()
    from gradient_compression_ef_gb300 import gc
    r = np.random.default_rng(77)
    big = (100.0 * r.standard_normal(MAX_N)).astype(np.float32)
    small = r.standard_normal(1000).astype(np.float32)
    with gc.Context(MAX_N) as ctx:
        _compare(torch, gc, ctx, big, np.zeros(MAX_N, np.float32), MAX_N // 50, "large")
        _compare(torch, gc, ctx, small, (0.1 * small).astype(np.float32), 13, "small after large")
        _compare(torch, gc, ctx, small[:5], None, 5, "tiny, k = n")


def test_noalloc_allocates_nothing():
    """After a first call (which looks up the array's address), further calls
    change neither the device's free memory nor torch's allocator."""
    torch = torch_cuda()
    from gradient_compression_ef_gb300 import gc
    r = np.random.default_rng(5)
    n, k = 500_000, 5_000
    gd = dev_f32(torch, r.standard_normal(n).astype(np.float32))
    ed = dev_f32(torch, np.zeros(n, np.float32))
    idx, val = _outputs(torch, k)
    _noalloc(gc, torch, gd, ed, n, k, idx, val)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    stats0 = torch.cuda.memory_stats()
    for _ in range(5):
        _noalloc(gc, torch, gd, ed, n, k, idx, val)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    stats1 = torch.cuda.memory_stats()
    assert free1 == free0
    for key in ("allocation.all.allocated", "segment.all.allocated", "reserved_bytes.all.current"):
        assert stats1.get(key) == stats0.get(key), key


def test_noalloc_rejects_sizes_above_its_maximum():
    torch = torch_cuda()
    from gradient_compression_ef_gb300 import gc
    n = gc.NOALLOC_MAX_N + 1
    g = torch.zeros(n, dtype=torch.float32, device="cuda")
    idx = torch.zeros(4, dtype=torch.int32, device="cuda")
    val = torch.zeros(4, dtype=torch.float32, device="cuda")
    with pytest.raises(gc.GCError) as ei:
        gc.ef_topk_noalloc(g, None, 4, idx, val)
    assert ei.value.status == gc.ERR_WORKSPACE
