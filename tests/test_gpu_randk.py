"""Random sparsification with error feedback on the GPU against the oracle,
bit for bit ('分布式训练中的梯度压缩算法' 二.2 随机稀疏化)."""
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
    ctx = gc.Context(1 << 21)
    yield torch, gc, ctx
    ctx.close()


def run(env, g, e, p, seed, step, capacity=None):
    torch, gc, ctx = env
    n = g.size
    cap = n if capacity is None else capacity
    gd = dev_f32(torch, g)
    ed = dev_f32(torch, e) if e is not None else None
    idx = torch.full((max(cap, 4),), -1, dtype=torch.int32, device="cuda")
    val = torch.full((max(cap, 4),), -1.0, dtype=torch.float32, device="cuda")
    cnt = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    gc.ef_randk(ctx, gd, ed, p, seed, step, idx, val, cnt, n=n, capacity=cap)
    return host(idx), host(val), (host(ed) if ed is not None else None), int(host(cnt)[0])


@pytest.mark.parametrize("n", [1, 5, 2048, 4097, 100_003, 1 << 20])
@pytest.mark.parametrize("p", [0.0, 0.01, 0.3, 1.0])
@pytest.mark.parametrize("ef", [True, False])
def test_matches_oracle(env, n, p, ef):
    r = np.random.default_rng(n)
    g = r.standard_normal(n).astype(np.float32)
    e = (0.1 * r.standard_normal(n)).astype(np.float32) if ef else None
    idx, val, e2, cnt = run(env, g, e, p, 17, 3)
    env[2].check()
    o_idx, o_val, o_err = oracle.ef_randk(g, None if e is None else e.copy(), p, 17, 3)
    assert cnt == o_idx.size
    assert_bits_equal(idx[:cnt], o_idx, "idx")
    assert_bits_equal(val[:cnt], o_val, "val")
    if ef:
        assert_bits_equal(e2, o_err, "err")


def test_capacity_overflow_is_flagged(env):
    torch, gc, ctx = env
    r = np.random.default_rng(1)
    g = r.standard_normal(50_000).astype(np.float32)
    o_idx, o_val, _ = oracle.ef_randk(g, None, 0.1, 5, 0)
    cap = o_idx.size // 2
    idx, val, _, cnt = run(env, g, None, 0.1, 5, 0, capacity=cap)
    with pytest.raises(gc.GCError) as ex:
        ctx.check()
    assert ex.value.status == gc.ERR_DEVICE_CHECK
    assert cnt == o_idx.size
    assert_bits_equal(idx[:cap], o_idx[:cap], "idx prefix")
    assert_bits_equal(val[:cap], o_val[:cap], "val prefix")


def test_leaves_the_context_clean_for_top_k(env):
    """A Top-K call on the same context after random sparsification gives
    the oracle's result (the scratch they share is left as Top-K needs it)."""
    torch, gc, ctx = env
    r = np.random.default_rng(2)
    g = r.standard_normal(300_000).astype(np.float32)
    run(env, g, np.zeros_like(g), 0.05, 1, 1)
    gd, ed = dev_f32(torch, g), dev_f32(torch, np.zeros_like(g))
    k = 3000
    idx = torch.empty(k, dtype=torch.int32, device="cuda")
    val = torch.empty(k, dtype=torch.float32, device="cuda")
    gc.ef_topk(ctx, gd, ed, k, idx, val)
    ctx.check()
    o_idx, o_val, o_err = oracle.ef_topk(g, np.zeros_like(g), k)
    assert_bits_equal(host(idx), o_idx, "topk idx")
    assert_bits_equal(host(ed), o_err, "topk err")


def test_full_size(env):
    """The 134,217,728-element gradient at p = 1 %, error feedback."""
    torch, gc, _ = env
    n = inputs.FLAT_ELEMS
    ctx = gc.Context(n)
    g = inputs.student_t_device(n, "cuda", seed=8)
    e = inputs.student_t_device(n, "cuda", seed=9).mul_(0.1)
    g_h, e_h = host(g), host(e)
    cap = n // 50
    idx = torch.empty(cap, dtype=torch.int32, device="cuda")
    val = torch.empty(cap, dtype=torch.float32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    gc.ef_randk(ctx, g, e, 0.01, 123, 4, idx, val, cnt)
    ctx.check()
    o_idx, o_val, o_err = oracle.ef_randk(g_h, e_h, 0.01, 123, 4)
    c = int(host(cnt)[0])
    assert c == o_idx.size
    assert_bits_equal(host(idx)[:c], o_idx, "full idx")
    assert_bits_equal(host(val)[:c], o_val, "full val")
    assert_bits_equal(host(e), o_err, "full err")
    ctx.close()


def test_validation(env):
    torch, gc, ctx = env
    x = torch.zeros(64, device="cuda")
    i = torch.zeros(64, dtype=torch.int32, device="cuda")
    c = torch.zeros(1, dtype=torch.int64, device="cuda")
    for p in (-0.1, 1.5, float("nan")):
        with pytest.raises(gc.GCError) as ex:
            gc.ef_randk(ctx, x, x, p, 0, 0, i, x, c)
        assert ex.value.status == gc.ERR_INVALID_ARG
    small = gc.Context(16)
    with pytest.raises(gc.GCError) as ex:
        gc.ef_randk(small, x, x, 0.5, 0, 0, i, x, c)
    assert ex.value.status == gc.ERR_WORKSPACE
    small.close()
