"""Pins of the oracle's aggregation of several ranks' compressed gradients
('分布式训练中的梯度压缩算法' 四: compress, aggregate, decompress): hand-worked
cases, numpy's own scatter-add applied rank by rank, and an independent
numpy decode of the QSGD codes."""
import json
import os

import numpy as np
import pytest

import oracle


def _load(golden_dir):
    return json.load(open(os.path.join(golden_dir, "aggregate_hand.json")))


def test_hand_cases(golden_dir):
    for case in _load(golden_dir)["cases"]:
        W, k, n = case["W"], case["k"], case["n"]
        out = oracle.topk_aggregate(np.array(case["idx"], np.int32),
                                    np.array(case["val"], np.float32), W, k, n)
        assert out.tolist() == case["out"], case["name"]
        assert not np.any(np.signbit(out[np.array(case["out"]) == 0.0])), case["name"]


def _pack(codes, signs, bits, k):
    """The documented layout, built with numpy: b-bit codes LSB-first padded
    to 16 bytes, then the sign plane padded to 16 bytes."""
    cbits = np.zeros(k * bits, np.uint8)
    for j, c in enumerate(codes):
        for b in range(bits):
            cbits[j * bits + b] = (c >> b) & 1
    mag = np.packbits(cbits, bitorder="little")
    mag = np.concatenate([mag, np.zeros(-(-mag.size // 16) * 16 - mag.size, np.uint8)])
    sg = np.packbits(np.array(signs, np.uint8), bitorder="little")
    sg = np.concatenate([sg, np.zeros(-(-sg.size // 16) * 16 - sg.size, np.uint8)])
    return np.concatenate([mag, sg])


def test_quant_hand_case(golden_dir):
    for case in _load(golden_dir)["quant_cases"]:
        W, k, n, bits, group = case["W"], case["k"], case["n"], case["bits"], case["group"]
        codes = np.concatenate([_pack(c, s, bits, k) for c, s in zip(case["codes"], case["signs"])])
        assert codes.size == W * oracle.codes_bytes(k, bits, "qsgd")
        scales = np.array([sc + [0.0] * (-len(sc) % 4) for sc in case["scales"]], np.float32)
        out = oracle.topk_quant_aggregate(np.array(case["idx"], np.int32), codes, scales, W, k,
                                          bits, group, n)
        assert out.tolist() == case["out"], case["name"]


def _ranks(r, W, k, n):
    return np.stack([np.sort(r.choice(n, size=k, replace=False)) for _ in range(W)]).astype(
        np.int32)


@pytest.mark.parametrize("W,k,n", [(1, 50, 200), (4, 300, 1000), (8, 1000, 1500), (3, 0, 10)])
def test_equals_numpy_scatter_add_in_rank_order(W, k, n):
    r = np.random.default_rng(W * 1000 + k)
    idx = _ranks(r, W, k, n)
    val = r.standard_normal((W, k)).astype(np.float32)
    want = np.zeros(n, np.float32)
    for w in range(W):  # float32 additions, rank by rank
        np.add.at(want, idx[w], val[w])
    got = oracle.topk_aggregate(idx, val, W, k, n)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    if W == 1:
        scat = np.zeros(n, np.float32)
        scat[idx[0]] = val[0]
        assert np.array_equal(got, scat)


@pytest.mark.parametrize("bits,group", [(8, 64), (4, 16), (2, 4), (1, 128)])
def test_quant_equals_numpy_decode_then_scatter(bits, group):
    """The quantised aggregate equals the plain aggregate of values decoded
    here with numpy from the documented code layout."""
    r = np.random.default_rng(bits * 7 + group)
    W, k, n = 3, 257, 2000
    idx = _ranks(r, W, k, n)
    top = (1 << bits) - 1
    q = r.integers(0, top + 1, size=(W, k))
    sg = (r.random((W, k)) < 0.5) & (q != 0)
    ng = -(-k // group)
    scales = (r.random((W, -(-ng // 4) * 4)) + 0.1).astype(np.float32)  # 16-byte rank stride
    codes = np.concatenate([_pack(q[w], sg[w], bits, k) for w in range(W)])
    vals = np.zeros((W, k), np.float32)
    for w in range(W):
        s = scales[w][np.arange(k) // group]
        m = (q[w].astype(np.float32) * s).astype(np.float32)
        vals[w] = np.where(sg[w], -m, m)
    want = oracle.topk_aggregate(idx, vals, W, k, n)
    got = oracle.topk_quant_aggregate(idx, codes, scales, W, k, bits, group, n)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_rejects_bad_indices():
    val = np.ones((2, 2), np.float32)
    with pytest.raises(oracle.OracleError):  # not increasing
        oracle.topk_aggregate(np.array([[1, 0], [0, 1]], np.int32), val, 2, 2, 4)
    with pytest.raises(oracle.OracleError):  # out of range
        oracle.topk_aggregate(np.array([[0, 4], [0, 1]], np.int32), val, 2, 2, 4)
    with pytest.raises(oracle.OracleError):  # repeated
        oracle.topk_aggregate(np.array([[1, 1], [0, 1]], np.int32), val, 2, 2, 4)
