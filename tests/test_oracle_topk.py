"""Pins of the oracle's EF + Top-K against things other than itself:
hand-worked cases, brute force on tiny inputs, invariants, and the pages'
own library calls (np.argpartition, torch.topk, np.sort threshold) on inputs
where those calls are unambiguous."""
import json
import os

import numpy as np
import pytest

import oracle
from gradient_compression_ef_gb300 import inputs


def _case_arrays(case):
    return (np.array(case["grad"], np.float32), np.array(case["err"], np.float32),
            case["k"])


def test_hand_cases(golden_dir):
    data = json.load(open(os.path.join(golden_dir, "topk_hand.json")))
    for case in data["cases"]:
        g, e, k = _case_arrays(case)
        idx, val, e2 = oracle.ef_topk(g, e, k)
        assert idx.tolist() == case["idx"], case["name"]
        assert val.tolist() == case["val"], case["name"]
        assert e2.tolist() == case["err_out"], case["name"]
        kept = set(case["idx"])
        for i in kept:  # kept residuals are +0, not -0
            assert np.signbit(e2[i]) == False, case["name"]  # noqa: E712


def _brute(c, k):
    order = sorted(range(len(c)), key=lambda i: (-abs(float(c[i])), i))
    return sorted(order[:k])


@pytest.mark.parametrize("seed", range(40))
def test_brute_force_tiny(seed):
    r = np.random.default_rng(seed)
    n = int(r.integers(1, 70))
    # few distinct magnitudes so that ties are common
    g = (r.integers(-4, 5, size=n) * 0.5).astype(np.float32)
    e = (r.integers(-2, 3, size=n) * 0.25).astype(np.float32)
    for k in sorted({0, 1, n // 3, n - 1 if n > 1 else 0, n}):
        idx, val, e2 = oracle.ef_topk(g, e, k)
        c = g + e
        want = _brute(c, k)
        assert idx.tolist() == want
        assert np.array_equal(val, c[want])
        ref = c.copy()
        ref[want] = 0.0
        assert np.array_equal(e2.view(np.uint32), (ref + np.float32(0)).view(np.uint32)) or \
            np.array_equal(e2, ref)


@pytest.mark.parametrize("n,k", [(1000, 10), (4096, 41), (10007, 1), (5000, 4999)])
def test_invariants(n, k):
    r = np.random.default_rng(n + k)
    g = r.standard_normal(n).astype(np.float32)
    e = (0.1 * r.standard_normal(n)).astype(np.float32)
    idx, val, e2 = oracle.ef_topk(g, e, k)
    c = g + e
    assert idx.size == k and np.all(np.diff(idx) > 0)
    assert np.array_equal(val.view(np.uint32), c[idx].view(np.uint32))
    kept = np.zeros(n, bool)
    kept[idx] = True
    assert np.all(e2[kept] == 0) and not np.any(np.signbit(e2[kept]))
    assert np.array_equal(e2[~kept].view(np.uint32), c[~kept].view(np.uint32))
    # every kept |c| >= every dropped |c|
    if 0 < k < n:
        assert np.abs(val).min() >= np.abs(c[~kept]).max()
    # the multiset {val} + {e'_i : i dropped} is the multiset {c_i}, bitwise
    both = np.concatenate([val, e2[~kept]]).view(np.uint32)
    assert np.array_equal(np.sort(both), np.sort(c.view(np.uint32)))


def test_matches_page_library_calls():
    """Without ties, the kept set equals what the pages' own calls return:
    np.argpartition (分布式训练中的梯度压缩算法 二.2), torch.topk
    (4、梯度累积与梯度压缩 4.2.1) and np.sort threshold with >= (梯度聚合通信
    优化实战方案 Python 演示)."""
    torch = pytest.importorskip("torch")
    r = np.random.default_rng(3)
    n = 20000
    # distinct magnitudes by construction: a shuffled ramp with random signs
    c = ((r.permutation(n) + 1) * r.choice([-1.0, 1.0], size=n)).astype(np.float32)
    c *= np.float32(2.0 ** -10)
    assert np.unique(np.abs(c)).size == n
    for k in (1, 200, 1999):
        idx, _, _ = oracle.ef_topk(c, None, k)
        part = np.sort(np.argpartition(np.abs(c), -k)[-k:])
        tk = np.sort(torch.topk(torch.from_numpy(np.abs(c)), k).indices.numpy())
        thr = np.sort(np.abs(c))[-k]
        demo = np.where(np.abs(c) >= thr)[0]
        assert idx.tolist() == part.tolist() == tk.tolist() == demo.tolist()


def test_demo_two_steps():
    """The Python demo's error-feedback replay at 1 % (k = 10,000): step 2
    runs on 0.9 * grad with the residual of step 1."""
    g = inputs.demo_gradient()
    k = inputs.ratio_k(g.size, 1, 100)
    assert k == 10_000
    e0 = np.zeros_like(g)
    idx1, val1, e1 = oracle.ef_topk(g, e0, k)
    g2 = g * np.float32(0.9)
    idx2, val2, e2 = oracle.ef_topk(g2, e1, k)
    c2 = g2 + e1
    assert np.array_equal(val2, c2[idx2])
    # step 1 residual is the gradient with the top 1 % removed
    assert np.abs(val1).min() >= np.abs(e1).max()
    # error energy of step 2 exceeds step 1 (residual accumulates)
    assert float(np.sum(e2.astype(np.float64) ** 2)) > \
        float(np.sum(e1.astype(np.float64) ** 2))
    # compression ratio of the sparse format with int32 indices: 4n / 8k
    assert (4 * g.size) / (idx1.nbytes + val1.nbytes) == 50.0


def test_no_residual_when_err_is_none():
    g = np.array([3, -5, 1], np.float32)
    idx, val, e = oracle.ef_topk(g, None, 1)
    assert e is None and idx.tolist() == [1] and val.tolist() == [-5]


def test_rejects_bad_k():
    with pytest.raises(oracle.OracleError):
        oracle.ef_topk(np.ones(4, np.float32), None, 5)
