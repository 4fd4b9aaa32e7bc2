"""gc_ef_topk_noalloc -- the allocation-free EF + Top-K entry point.

Some callers cannot allocate device memory (their memory belongs to another
allocator, or they run under a hard budget or on a path where cudaMalloc's
device-wide synchronisation is not acceptable), so they cannot create a
context.  This entry point keeps its scratch in a static device array of the
library instead.  Here it is called through the C ABI twice in a row (two
error-feedback steps) and must give exactly what gc_ef_topk with a context
gives on the same inputs.  This file is collected last on purpose.
"""
import numpy as np
import pytest

from tests.gpu_helpers import assert_bits_equal, dev_f32, host, torch_cuda

pytestmark = pytest.mark.gpu


def _outputs(torch, k):
    return (torch.full((k,), -1, dtype=torch.int32, device="cuda"),
            torch.full((k,), -1.0, dtype=torch.float32, device="cuda"))


def test_noalloc_matches_context_call_on_two_calls_in_a_row():
    torch = torch_cuda()
    from gradient_compression_ef_gb300 import gc
    r = np.random.default_rng(20261202)
    n, k = 1_000_003, 10_000
    g1 = r.standard_normal(n).astype(np.float32)
    g2 = r.standard_normal(n).astype(np.float32)
    e0 = (0.1 * r.standard_normal(n)).astype(np.float32)

    e_ctx, e_na = dev_f32(torch, e0), dev_f32(torch, e0)
    stream = torch.cuda.current_stream()
    with gc.Context(n) as ctx:
        for step, g in enumerate((g1, g2)):
            gd = dev_f32(torch, g)
            i_ctx, v_ctx = _outputs(torch, k)
            gc.ef_topk(ctx, gd, e_ctx, k, i_ctx, v_ctx)
            ctx.check()
            i_na, v_na = _outputs(torch, k)
            st = gc.lib.gc_ef_topk_noalloc(gd.data_ptr(), e_na.data_ptr(), n, k,
                                           i_na.data_ptr(), v_na.data_ptr(),
                                           stream.cuda_stream)
            assert st == gc.OK, gc.status_string(st)
            torch.cuda.synchronize()
            what = "call %d" % (step + 1)
            assert_bits_equal(host(i_na), host(i_ctx), what + " idx")
            assert_bits_equal(host(v_na), host(v_ctx), what + " val")
            assert_bits_equal(host(e_na), host(e_ctx), what + " err")


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
