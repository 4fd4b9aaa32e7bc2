"""Aggregation of several ranks' compressed gradients on the GPU against the
oracle, bit for bit ('分布式训练中的梯度压缩算法' 四: compress, aggregate,
decompress)."""
import json
import os

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
    ctx = gc.Context(1 << 20)
    yield torch, gc, ctx
    ctx.close()


def ranks(r, W, k, n):
    return np.stack([np.sort(r.choice(n, size=k, replace=False)) for _ in range(W)]).astype(
        np.int32).reshape(W, k)


def padded(a, W, k, dtype):
    """(W, k) rows in the device layout: rank w at w * K, K = k rounded up to 4."""
    K = -(-k // 4) * 4
    out = np.zeros((W, max(K, 1)), dtype=dtype)
    out[:, :k] = np.asarray(a, dtype=dtype).reshape(W, k)
    return out.reshape(-1)


def run_plain(env, idx, val, W, k, n):
    torch, gc, ctx = env
    out = torch.full((max(n, 4),), 7.0, dtype=torch.float32, device="cuda")
    di = torch.from_numpy(padded(idx, W, k, np.int32)).cuda()
    dv = dev_f32(torch, padded(val, W, k, np.float32))
    gc.topk_aggregate(ctx, W, k, di, dv, n, out)
    ctx.check()
    return host(out)[:n]


@pytest.mark.parametrize("W,k,n", [(1, 100, 1000), (3, 5000, 30001), (8, 2000, 8192),
                                   (8, 9000, 100_003), (16, 300, 7), (2, 0, 5000),
                                   (5, 1, 1), (40, 700, 50_000), (33, 4000, 4096)])
def test_random_ranks(env, W, k, n):
    k = min(k, n)
    r = np.random.default_rng(W * 31 + k)
    idx = ranks(r, W, k, n)
    val = r.standard_normal((W, k)).astype(np.float32)
    got = run_plain(env, idx, val, W, k, n)
    assert_bits_equal(got, oracle.topk_aggregate(idx, val, W, k, n), "W=%d k=%d n=%d" % (W, k, n))


def test_dense_ranks_take_several_chunks(env):
    """Every rank keeps every element: one output range receives 3 x 8192
    entries, more than one gathering chunk holds."""
    W, n = 3, 20000
    idx = np.tile(np.arange(n, dtype=np.int32), (W, 1))
    r = np.random.default_rng(5)
    val = (r.standard_normal((W, n)) * np.array([[1e8], [1.0], [-1e8]])).astype(np.float32)
    got = run_plain(env, idx, val, W, n, n)
    assert_bits_equal(got, oracle.topk_aggregate(idx, val, W, n, n), "dense")


def clustered_ranks(r, W, k, n):
    """Ranks of mixed density: rank w draws its k indices from a window of
    2k, 5k, n / 2 or n elements (by w mod 4) at a random offset, so some
    ranks have hundreds of entries in a 1024-element range where others
    have a few, in the same group of ranks."""
    rows = []
    for w in range(W):
        span = min(n, (2 * k, 5 * k, n // 2, n)[w % 4])
        lo = int(r.integers(0, n - span + 1))
        rows.append(np.sort(lo + r.choice(span, size=k, replace=False)))
    return np.stack(rows).astype(np.int32)


@pytest.mark.parametrize("W,k,n", [(11, 3000, 200_000), (37, 2500, 120_000), (8, 600, 4096)])
def test_ranks_of_mixed_density(env, W, k, n):
    r = np.random.default_rng(W + 7 * k)
    idx = clustered_ranks(r, W, k, n)
    val = r.standard_normal((W, k)).astype(np.float32)
    got = run_plain(env, idx, val, W, k, n)
    assert_bits_equal(got, oracle.topk_aggregate(idx, val, W, k, n),
                      "mixed W=%d k=%d n=%d" % (W, k, n))


@pytest.mark.parametrize("bits,group", [(8, 48), (2, 100), (4, 0), (1, 7)])
def test_quant_ranks_any_group(env, bits, group):
    """Codes and scales drawn at random (the aggregation takes any bytes),
    groups that are not a power of two (a division per entry) or one group
    of all k, ranks of mixed density."""
    torch, gc, ctx = env
    W, n, k = 13, 150_000, 2000
    r = np.random.default_rng(bits * 1000 + group)
    idx = clustered_ranks(r, W, k, n)
    cb = gc.codes_bytes(k, bits, "qsgd")
    sf = -(-gc.scales_floats(k, group, "qsgd") // 4) * 4
    codes = r.integers(0, 256, size=W * cb, dtype=np.uint8)
    scales = r.uniform(0.5, 2.0, size=W * sf).astype(np.float32)
    out = torch.full((n,), 7.0, dtype=torch.float32, device="cuda")
    di = torch.from_numpy(padded(idx, W, k, np.int32)).cuda()
    gc.topk_quant_aggregate(ctx, W, k, di, torch.from_numpy(codes).cuda(),
                            dev_f32(torch, scales), bits, group, n, out)
    ctx.check()
    want = oracle.topk_quant_aggregate(idx, codes, scales, W, k, bits, group, n)
    assert_bits_equal(host(out), want, "bits=%d group=%d" % (bits, group))


def test_hand_cases(env, golden_dir):
    data = json.load(open(os.path.join(golden_dir, "aggregate_hand.json")))
    for case in data["cases"]:
        W, k, n = case["W"], case["k"], case["n"]
        got = run_plain(env, np.array(case["idx"], np.int32), np.array(case["val"], np.float32),
                        W, k, n)
        assert got.tolist() == case["out"], case["name"]


def compress_ranks(env, W, n, k, bits, group, seed):
    """W simulated ranks each compress their own gradient with the hybrid."""
    torch, gc, ctx = env
    cb = gc.codes_bytes(k, bits, "qsgd")
    sf = -(-gc.scales_floats(k, group, "qsgd") // 4) * 4  # rank stride: 16 bytes
    K = -(-k // 4) * 4
    idx = torch.zeros(W * K, dtype=torch.int32, device="cuda")
    codes = torch.empty(W * cb, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(max(W * sf, 4), dtype=torch.float32, device="cuda")
    for w in range(W):
        g = torch.from_numpy(inputs.student_t(inputs.rng(seed + w), n)).cuda()
        e = torch.zeros(n, dtype=torch.float32, device="cuda")
        gc.ef_topk_quant(ctx, g, e, k, bits, group, "stochastic", 3 + w, 0,
                         idx[w * K:w * K + k], codes[w * cb:(w + 1) * cb],
                         scales[w * sf:w * sf + gc.scales_floats(k, group, "qsgd")])
    ctx.check()
    return idx, codes, scales[:W * sf]


@pytest.mark.parametrize("bits,group", [(8, 64), (4, 16), (2, 128), (1, 4)])
def test_quant_ranks(env, bits, group):
    torch, gc, ctx = env
    W, n, k = 4, 100_000, 1000
    idx, codes, scales = compress_ranks(env, W, n, k, bits, group, 40 + bits)
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    gc.topk_quant_aggregate(ctx, W, k, idx, codes, scales, bits, group, n, out)
    ctx.check()
    K = -(-k // 4) * 4
    want = oracle.topk_quant_aggregate(host(idx).reshape(W, K)[:, :k], host(codes), host(scales),
                                       W, k, bits, group, n)
    assert_bits_equal(host(out), want, "bits=%d group=%d" % (bits, group))


def test_full_size_eight_ranks(env):
    """Eight ranks' Top-K 1 % + 8-bit QSGD outputs over a 134,217,728-element
    gradient aggregated into one dense buffer."""
    torch, gc, _ = env
    W, n = 8, inputs.FLAT_ELEMS
    k = inputs.ratio_k(n, 1, 100)
    ctx = gc.Context(n)
    cb = gc.codes_bytes(k, 8, "qsgd")
    sf = -(-gc.scales_floats(k, 64, "qsgd") // 4) * 4
    K = -(-k // 4) * 4
    idx = torch.zeros(W * K, dtype=torch.int32, device="cuda")
    codes = torch.empty(W * cb, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(W * sf, dtype=torch.float32, device="cuda")
    e = torch.zeros(n, dtype=torch.float32, device="cuda")
    for w in range(W):
        g = inputs.student_t_device(n, "cuda", seed=100 + w)
        e.zero_()
        gc.ef_topk_quant(ctx, g, e, k, 8, 64, "stochastic", 9 + w, 0, idx[w * K:w * K + k],
                         codes[w * cb:(w + 1) * cb],
                         scales[w * sf:w * sf + gc.scales_floats(k, 64, "qsgd")])
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    gc.topk_quant_aggregate(ctx, W, k, idx, codes, scales, 8, 64, n, out)
    ctx.check()
    want = oracle.topk_quant_aggregate(host(idx).reshape(W, K)[:, :k], host(codes), host(scales),
                                       W, k, 8, 64, n)
    assert_bits_equal(host(out), want, "full size")
    ctx.close()


def test_validation(env):
    torch, gc, ctx = env
    i = torch.zeros(16, dtype=torch.int32, device="cuda")
    v = torch.zeros(16, dtype=torch.float32, device="cuda")
    o = torch.zeros(64, dtype=torch.float32, device="cuda")
    for W, k, n, status in ((0, 1, 8, gc.ERR_INVALID_ARG), (2000, 1, 8, gc.ERR_INVALID_ARG),
                            (1, 9, 8, gc.ERR_INVALID_ARG)):
        with pytest.raises(gc.GCError) as ex:
            gc.topk_aggregate(ctx, W, k, i, v, n, o)
        assert ex.value.status == status
    small = gc.Context(16)
    with pytest.raises(gc.GCError) as ex:
        gc.topk_aggregate(small, 4, 1, i, v, 1 << 20, o)
    assert ex.value.status == gc.ERR_WORKSPACE
    small.close()
    with pytest.raises(gc.GCError) as ex:
        gc.topk_quant_aggregate(ctx, 1, 4, i, o, v, 3, 64, 8, o)
    assert ex.value.status == gc.ERR_UNSUPPORTED


def test_bad_indices_are_flagged(env):
    """Indices that are not strictly increasing or out of range set the
    device status; nothing is read or written out of bounds."""
    torch, gc, ctx = env
    n = 50
    for bad in ([3, 3, 9], [9, 3, 12], [1, 2, 50], [-1, 4, 7]):
        idx = torch.tensor(bad, dtype=torch.int32, device="cuda")
        val = torch.ones(3, dtype=torch.float32, device="cuda")
        out = torch.zeros(n, dtype=torch.float32, device="cuda")
        gc.topk_aggregate(ctx, 1, 3, idx, val, n, out)
        with pytest.raises(gc.GCError) as ex:
            ctx.check()
        assert ex.value.status == gc.ERR_DEVICE_CHECK
