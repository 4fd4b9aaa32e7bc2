"""Robustness on the GPU: guard zones around every output (no call writes
outside its buffers), allocation failure reported as a status with the
context still usable, and checkpoint / resume of the compressor's state
(error buffer, PowerSGD's Q) into a fresh context giving bit-identical
results."""
import numpy as np
import pytest

from gradient_compression_ef_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, dev_f32, host, torch_cuda

pytestmark = pytest.mark.gpu

GUARD = 64          # bytes of 0xCD before and after each output
PATTERN = 0xCD


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from gradient_compression_ef_gb300 import gc
    ctx = gc.Context(1 << 20)
    ctx.reserve_powersgd(512, 512, 8)
    yield torch, gc, ctx
    ctx.close()


class Guarded:
    """A device buffer of `count` elements of `dtype` between two guard
    zones; `t` is the (16-byte aligned) view the call writes."""

    def __init__(self, torch, count, dtype, fill=None):
        itemsize = torch.empty(0, dtype=dtype).element_size()
        nbytes = max(count, 1) * itemsize
        self.raw = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + nbytes].view(dtype)[:max(count, 1)]
        if fill is not None:
            self.t.copy_(fill)

    def intact(self):
        r = host(self.raw)
        return bool(np.all(r[:GUARD] == PATTERN) and np.all(r[-GUARD:] == PATTERN))


def check_guards(bufs, what):
    for name, b in bufs.items():
        assert b.intact(), "%s: guard zone of %s overwritten" % (what, name)


def test_guard_zones_of_every_call(env):
    torch, gc, ctx = env
    f32, i32, u8 = torch.float32, torch.int32, torch.uint8
    r = np.random.default_rng(0)
    n, k = 10_007, 101
    g = torch.from_numpy(r.standard_normal(n).astype(np.float32)).cuda()
    # Top-K
    b = {"err": Guarded(torch, n, f32, fill=g * 0.1), "idx": Guarded(torch, k, i32),
         "val": Guarded(torch, k, f32)}
    gc.ef_topk(ctx, g, b["err"].t, k, b["idx"].t, b["val"].t)
    ctx.check()
    check_guards(b, "ef_topk")
    # quantisation, every mode, fused and multi-pass groups, and dequantisation
    for mode, bits in (("minmax", 1), ("minmax", 4), ("qsgd", 8), ("qsgd", 2), ("tern", 2),
                       ("log", 4)):
        for group in (64, 100, 0):
            b = {"err": Guarded(torch, n, f32, fill=g * 0.1),
                 "codes": Guarded(torch, gc.codes_bytes(n, bits, mode), u8),
                 "scales": Guarded(torch, gc.scales_floats(n, group, mode), f32),
                 "out": Guarded(torch, n, f32)}
            gc.ef_quant(ctx, g, b["err"].t, bits, group, mode, "stochastic", 1, 2, b["codes"].t,
                        b["scales"].t)
            gc.dequant(ctx, b["codes"].t, b["scales"].t, n, bits, group, mode, b["out"].t)
            ctx.check()
            check_guards(b, "quant %s/%d g%d" % (mode, bits, group))
    # hybrid single call
    b = {"err": Guarded(torch, n, f32, fill=g * 0.1), "idx": Guarded(torch, k, i32),
         "codes": Guarded(torch, gc.codes_bytes(k, 8, "qsgd"), u8),
         "scales": Guarded(torch, gc.scales_floats(k, 64, "qsgd"), f32)}
    gc.ef_topk_quant(ctx, g, b["err"].t, k, 8, 64, "stochastic", 3, 4, b["idx"].t, b["codes"].t,
                     b["scales"].t)
    ctx.check()
    check_guards(b, "ef_topk_quant")
    # bucketed hybrid with diagnostics
    ns, ks = [4096, 2048, 3863], [41, 2048, 0]
    ctx.set_buckets(ns, ks)
    oi, oc, os_ = gc.bucket_offsets(ks, 4, 16)
    b = {"err": Guarded(torch, n, f32, fill=g * 0.1), "idx": Guarded(torch, oi[-1], i32),
         "codes": Guarded(torch, oc[-1], u8), "scales": Guarded(torch, os_[-1], f32),
         "diag": Guarded(torch, 3 * len(ns), torch.float64)}
    for step in range(2):
        gc.ef_topk_quant_buckets(ctx, g, b["err"].t, 4, 16, "stochastic", 5, step, b["idx"].t,
                                 b["codes"].t, b["scales"].t, diag=b["diag"].t)
    ctx.check()
    check_guards(b, "ef_topk_quant_buckets")
    # Random-K with a capacity below the kept count
    b = {"err": Guarded(torch, n, f32, fill=g * 0.1), "idx": Guarded(torch, 37, i32),
         "val": Guarded(torch, 37, f32), "count": Guarded(torch, 1, torch.int64)}
    gc.ef_randk(ctx, g, b["err"].t, 0.05, 7, 0, b["idx"].t, b["val"].t, b["count"].t,
                capacity=37)
    with pytest.raises(gc.GCError):
        ctx.check()  # more kept than the capacity: flagged, nothing written past it
    check_guards(b, "ef_randk")
    # differential quantisation and its receiving side
    b = {"err": Guarded(torch, n, f32, fill=g * 0.1), "ref": Guarded(torch, n, f32, fill=g),
         "codes": Guarded(torch, gc.codes_bytes(n, 4, "minmax"), u8),
         "scales": Guarded(torch, gc.scales_floats(n, 32, "minmax"), f32),
         "recv": Guarded(torch, n, f32, fill=g)}
    gc.ef_diff_quant(ctx, g, b["err"].t, b["ref"].t, 4, 32, "minmax", "nearest_even", 0, 1,
                     False, b["codes"].t, b["scales"].t)
    gc.diff_dequant(ctx, b["codes"].t, b["scales"].t, n, 4, 32, "minmax", False, b["recv"].t)
    ctx.check()
    check_guards(b, "diff")
    # aggregation of 3 ranks
    W, ka, na = 3, 50, 3001
    K = -(-ka // 4) * 4
    idx = np.zeros((W, K), np.int32)
    for w in range(W):
        idx[w, :ka] = np.sort(r.choice(na, ka, replace=False))
    b = {"out": Guarded(torch, na, f32)}
    gc.topk_aggregate(ctx, W, ka, torch.from_numpy(idx.reshape(-1)).cuda(),
                      torch.ones(W * K, device="cuda"), na, b["out"].t)
    ctx.check()
    check_guards(b, "topk_aggregate")
    # PowerSGD
    m, nn, rr = 300, 211, 3
    G = torch.randn(m * nn, device="cuda")
    b = {"err": Guarded(torch, m * nn, f32, fill=torch.zeros(m * nn, device="cuda")),
         "P": Guarded(torch, m * rr, f32), "Q": Guarded(torch, nn * rr, f32,
                                                      fill=torch.randn(nn * rr, device="cuda"))}
    gc.powersgd_step(ctx, G, b["err"].t, m, nn, rr, b["P"].t, b["Q"].t)
    ctx.check()
    check_guards(b, "powersgd_step")


def test_allocation_failure_is_a_status(env):
    """A plan too large for the device returns GC_ERR_NO_MEMORY; the context
    keeps working with a new plan."""
    torch, gc, _ = env
    ctx = gc.Context(0)
    with pytest.raises(gc.GCError) as ex:
        ctx.set_buckets([1 << 21] * 20_000, [1] * 20_000)  # ~340 GB of scratch
    assert ex.value.status == gc.ERR_NO_MEMORY
    with pytest.raises(gc.GCError) as ex:
        ctx.reserve_powersgd(1 << 30, 1 << 30, 16)
    assert ex.value.status == gc.ERR_NO_MEMORY
    ctx.set_buckets([4096], [40])
    g = torch.randn(4096, device="cuda")
    e = torch.zeros(4096, device="cuda")
    idx = torch.empty(40, dtype=torch.int32, device="cuda")
    val = torch.empty(40, device="cuda")
    gc.ef_topk_buckets(ctx, g, e, idx, val)
    ctx.check()
    assert np.array_equal(np.sort(np.abs(host(val))), np.sort(np.abs(host(g)))[-40:])
    ctx.close()


def test_checkpoint_resume_bucketed(env):
    """Ten correlated steps straight, against five steps, the residual copied
    to the host, a fresh context and plan, the residual restored, five more
    steps: outputs and residual bit-identical (the threshold guess a plan
    carries between calls never changes a result)."""
    torch, gc, _ = env
    ns = [65_536, 131_072, 30_001]
    ks = [655, 1_310, 300]
    n = sum(ns)
    grads = [dev_f32(torch, g) for g in inputs.correlated_steps(n, 10, seed=8)]
    oi, oc, os_ = gc.bucket_offsets(ks, 8, 64)

    def run(ctx, e, steps):
        outs = []
        for t in steps:
            idx = torch.empty(oi[-1], dtype=torch.int32, device="cuda")
            codes = torch.empty(oc[-1], dtype=torch.uint8, device="cuda")
            scales = torch.empty(os_[-1], dtype=torch.float32, device="cuda")
            gc.ef_topk_quant_buckets(ctx, grads[t], e, 8, 64, "stochastic", 77, t, idx, codes,
                                     scales)
            outs.append((host(idx), host(codes), host(scales)))
        ctx.check()
        return outs

    a = gc.Context(0)
    a.set_buckets(ns, ks)
    e_a = torch.zeros(n, device="cuda")
    straight = run(a, e_a, range(10))
    b = gc.Context(0)
    b.set_buckets(ns, ks)
    e_b = torch.zeros(n, device="cuda")
    run(b, e_b, range(5))
    saved = host(e_b).copy()
    b.close()
    c = gc.Context(0)
    c.set_buckets(ns, ks)
    e_c = dev_f32(torch, saved)
    resumed = run(c, e_c, range(5, 10))
    # the slots between buckets (padding to 16 bytes) are not written
    sf = [gc.scales_floats(kb, 64, "qsgd") for kb in ks]
    for t, (x, y) in enumerate(zip(straight[5:], resumed)):
        w = "step %d" % (t + 5)
        for bk in range(len(ks)):
            assert_bits_equal(y[0][oi[bk]:oi[bk] + ks[bk]], x[0][oi[bk]:oi[bk] + ks[bk]], w + " idx")
            assert_bits_equal(y[2][os_[bk]:os_[bk] + sf[bk]], x[2][os_[bk]:os_[bk] + sf[bk]],
                              w + " scales")
        assert_bits_equal(y[1], x[1], w + " codes")
    assert_bits_equal(host(e_c), host(e_a), "residual")
    a.close()
    c.close()


def test_checkpoint_resume_powersgd(env):
    """Four PowerSGD steps straight against two, (E, Q) restored into a fresh
    context, two more: bit-identical (the reductions have a fixed order)."""
    torch, gc, _ = env
    m, n, r = 1024, 768, 4
    M, Q0 = inputs.low_rank_matrix(m, n, seed=3, r=r)
    G = dev_f32(torch, M)

    def steps(ctx, E, Q, count):
        P = torch.empty(m * r, device="cuda")
        for _ in range(count):
            gc.powersgd_step(ctx, G, E, m, n, r, P, Q)
        ctx.check()
        return host(P)

    a = gc.Context(0)
    a.reserve_powersgd(m, n, r)
    Ea, Qa = torch.zeros(m * n, device="cuda"), dev_f32(torch, Q0)
    Pa = steps(a, Ea, Qa, 4)
    b = gc.Context(0)
    b.reserve_powersgd(m, n, r)
    Eb, Qb = torch.zeros(m * n, device="cuda"), dev_f32(torch, Q0)
    steps(b, Eb, Qb, 2)
    E_saved, Q_saved = host(Eb).copy(), host(Qb).copy()
    b.close()
    c = gc.Context(0)
    c.reserve_powersgd(m, n, r)
    Ec, Qc = dev_f32(torch, E_saved), dev_f32(torch, Q_saved)
    Pc = steps(c, Ec, Qc, 2)
    assert_bits_equal(Pc, Pa, "P")
    assert_bits_equal(host(Qc), host(Qa), "Q")
    assert_bits_equal(host(Ec), host(Ea), "E")
    a.close()
    c.close()
