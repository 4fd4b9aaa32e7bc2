"""Shared helpers of the GPU parity tests (bitwise comparisons, buffers)."""
import numpy as np
import pytest


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def dev_f32(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host(t):
    return t.cpu().numpy()


def assert_bits_equal(got, want, what):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, "%s: shape %s vs %s" % (what, got.shape, want.shape)
    if got.dtype == np.float32:
        g, w = got.view(np.uint32), want.astype(np.float32).view(np.uint32)
    else:
        g, w = got, want
    bad = np.nonzero(g != w)[0]
    assert bad.size == 0, "%s: %d mismatches, first at %d (got %r want %r)" % (
        what, bad.size, bad[0], got.ravel()[bad[0]], want.ravel()[bad[0]])
