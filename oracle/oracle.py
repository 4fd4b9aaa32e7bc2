"""NumPy front end of the C oracle (test infrastructure).

Each function copies its inputs, calls the single-threaded C statement of the
method in ``gc_oracle.c`` and returns fresh NumPy arrays.  Nothing here does
arithmetic of the method; it only marshals buffers.

Mode and rounding numbers are the oracle's own:
MINMAX = 0, QSGD = 1, TERN = 2; NEAREST_EVEN = 0, STOCHASTIC = 1.
"""
import ctypes
import os

import numpy as np

from . import build as _build

MINMAX, QSGD, TERN, LOG = 0, 1, 2, 3
NEAREST_EVEN, STOCHASTIC = 0, 1
MODES = {"minmax": MINMAX, "qsgd": QSGD, "tern": TERN, "log": LOG}
ROUNDINGS = {"nearest_even": NEAREST_EVEN, "stochastic": STOCHASTIC}

_lib = None

_f32p = ctypes.POINTER(ctypes.c_float)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64
_int = ctypes.c_int


class OracleError(RuntimeError):
    pass


def lib():
    """Loads (building first if needed) ``libgc_oracle.so``."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path) or (
                os.path.getmtime(path) < os.path.getmtime(_build.SRC)):
            _build.build()
        L = ctypes.CDLL(path)
        L.orc_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
        L.orc_philox4x32_10.restype = None
        L.orc_uniform.argtypes = [_u64, _u64, _u64]
        L.orc_uniform.restype = ctypes.c_float
        L.orc_bucket_seed.argtypes = [_u64, _i64]
        L.orc_bucket_seed.restype = _u64
        L.orc_codes_bytes.argtypes = [_i64, _int, _int]
        L.orc_codes_bytes.restype = _i64
        L.orc_scales_floats.argtypes = [_i64, _i64, _int]
        L.orc_scales_floats.restype = _i64
        L.orc_ef_topk.argtypes = [_f32p, _f32p, _i64, _i64, _i32p, _f32p]
        L.orc_ef_topk.restype = _int
        L.orc_quant.argtypes = [_f32p, _i64, _int, _i64, _int, _int, _u64,
                                _u64, _u8p, _f32p]
        L.orc_quant.restype = _int
        L.orc_quant_at.argtypes = [_f32p, _i64, _i64, _int, _i64, _int, _int,
                                   _u64, _u64, _u8p, _f32p]
        L.orc_quant_at.restype = _int
        L.orc_dequant.argtypes = [_u8p, _f32p, _i64, _int, _i64, _int, _f32p]
        L.orc_dequant.restype = _int
        L.orc_ef_quant.argtypes = [_f32p, _f32p, _i64, _int, _i64, _int, _int,
                                   _u64, _u64, _u8p, _f32p]
        L.orc_ef_quant.restype = _int
        L.orc_ef_topk_quant.argtypes = [_f32p, _f32p, _i64, _i64, _int, _i64,
                                        _int, _u64, _u64, _i32p, _u8p, _f32p]
        L.orc_ef_topk_quant.restype = _int
        L.orc_powersgd_step.argtypes = [_f32p, _f32p, _i64, _i64, _int, _f32p,
                                        _f32p]
        L.orc_powersgd_step.restype = _int
        L.orc_ef_randk.argtypes = [_f32p, _f32p, _i64, ctypes.c_float, _u64, _u64, _i32p,
                                   _f32p, _i64, ctypes.POINTER(_i64)]
        L.orc_ef_randk.restype = _int
        L.orc_logf.argtypes = [ctypes.c_float]
        L.orc_logf.restype = ctypes.c_float
        L.orc_expf.argtypes = [ctypes.c_float]
        L.orc_expf.restype = ctypes.c_float
        L.orc_ef_diff_quant.argtypes = [_f32p, _f32p, _f32p, _i64, _int, _i64, _int, _int,
                                        _u64, _u64, _int, _u8p, _f32p]
        L.orc_ef_diff_quant.restype = _int
        L.orc_diff_dequant.argtypes = [_u8p, _f32p, _i64, _int, _i64, _int, _int, _f32p]
        L.orc_diff_dequant.restype = _int
        L.orc_diagnostics.argtypes = [_f32p, _f32p, _i64, _i32p, _f32p, _i64,
                                      ctypes.POINTER(ctypes.c_double)]
        L.orc_diagnostics.restype = _int
        L.orc_topk_aggregate.argtypes = [_int, _i64, _i32p, _f32p, _i64, _f32p]
        L.orc_topk_aggregate.restype = _int
        L.orc_topk_quant_aggregate.argtypes = [_int, _i64, _i32p, _u8p, _f32p, _int, _i64,
                                               _i64, _f32p]
        L.orc_topk_quant_aggregate.restype = _int
        _lib = L
    return _lib


def _p(a, t):
    return a.ctypes.data_as(t) if a is not None else None


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32)).copy()


def _check(st, what):
    if st != 0:
        raise OracleError("%s failed with status %d" % (what, st))


def _mode(mode):
    return MODES[mode] if isinstance(mode, str) else int(mode)


def _rounding(r):
    return ROUNDINGS[r] if isinstance(r, str) else int(r)


def philox4x32_10(counter, key):
    """Philox-4x32-10 block: 4 counter words, 2 key words -> 4 words."""
    c = np.asarray(counter, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_p(c, _u32p), _p(k, _u32p), _p(out, _u32p))
    return out


def uniform(seed, step, i):
    """The stochastic-rounding draw u in [0, 1) of element i."""
    return float(lib().orc_uniform(seed, step, i))


def bucket_seed(seed, b):
    """The Philox key bucket b of a bucketed call draws with."""
    return int(lib().orc_bucket_seed(seed, b))


def codes_bytes(n, bits, mode):
    return int(lib().orc_codes_bytes(n, bits, _mode(mode)))


def scales_floats(n, group, mode):
    return int(lib().orc_scales_floats(n, group, _mode(mode)))


def ef_topk(grad, err, k):
    """EF + Top-K.  Returns (idx int32[k], val float32[k], err' or None)."""
    g = _f32(grad)
    e = _f32(err) if err is not None else None
    n = g.size
    idx = np.zeros(max(k, 1), dtype=np.int32)
    val = np.zeros(max(k, 1), dtype=np.float32)
    _check(lib().orc_ef_topk(_p(g, _f32p), _p(e, _f32p), n, k,
                             _p(idx, _i32p), _p(val, _f32p)), "orc_ef_topk")
    return idx[:k], val[:k], e


def quant(x, bits, group, mode, rounding="nearest_even", seed=0, step=0):
    """Quantise x.  Returns (codes uint8[codes_bytes], scales float32[...])."""
    xs = _f32(x)
    n = xs.size
    m = _mode(mode)
    cb = codes_bytes(n, bits, m)
    sf = scales_floats(n, group, m)
    if cb < 0 or sf < 0:
        raise OracleError("bad quantisation arguments")
    codes = np.zeros(max(cb, 1), dtype=np.uint8)
    scales = np.zeros(max(sf, 1), dtype=np.float32)
    _check(lib().orc_quant(_p(xs, _f32p), n, bits, group, m,
                           _rounding(rounding), seed, step, _p(codes, _u8p),
                           _p(scales, _f32p)), "orc_quant")
    return codes[:cb], scales[:sf]


def quant_at(x, base, bits, group, mode, rounding="nearest_even", seed=0,
             step=0):
    """quant() of a group-aligned slice that starts at element ``base`` of
    a larger call (the stochastic draws follow the call's indices)."""
    xs = _f32(x)
    n = xs.size
    m = _mode(mode)
    cb = codes_bytes(n, bits, m)
    sf = scales_floats(n, group, m)
    codes = np.zeros(max(cb, 1), dtype=np.uint8)
    scales = np.zeros(max(sf, 1), dtype=np.float32)
    _check(lib().orc_quant_at(_p(xs, _f32p), n, base, bits, group, m,
                              _rounding(rounding), seed, step,
                              _p(codes, _u8p), _p(scales, _f32p)),
           "orc_quant_at")
    return codes[:cb], scales[:sf]


def dequant(codes, scales, n, bits, group, mode):
    c = np.ascontiguousarray(codes, dtype=np.uint8).copy()
    s = _f32(scales)
    out = np.zeros(max(n, 1), dtype=np.float32)
    if c.size == 0:
        c = np.zeros(1, dtype=np.uint8)
    if s.size == 0:
        s = np.zeros(1, dtype=np.float32)
    _check(lib().orc_dequant(_p(c, _u8p), _p(s, _f32p), n, bits, group,
                             _mode(mode), _p(out, _f32p)), "orc_dequant")
    return out[:n]


def ef_quant(grad, err, bits, group, mode, rounding="nearest_even", seed=0,
             step=0):
    """EF + quantise.  Returns (codes, scales, err')."""
    g = _f32(grad)
    e = _f32(err)
    n = g.size
    m = _mode(mode)
    cb = codes_bytes(n, bits, m)
    sf = scales_floats(n, group, m)
    codes = np.zeros(max(cb, 1), dtype=np.uint8)
    scales = np.zeros(max(sf, 1), dtype=np.float32)
    _check(lib().orc_ef_quant(_p(g, _f32p), _p(e, _f32p), n, bits, group, m,
                              _rounding(rounding), seed, step,
                              _p(codes, _u8p), _p(scales, _f32p)),
           "orc_ef_quant")
    return codes[:cb], scales[:sf], e


def logf(x):
    """The oracle's binary32 natural logarithm (x >= 1)."""
    return np.float32(lib().orc_logf(float(x)))


def expf(y):
    """The oracle's binary32 exponential (0 <= y < 89)."""
    return np.float32(lib().orc_expf(float(y)))


def ef_diff_quant(grad, err, ref, bits, group, mode, rounding="nearest_even", seed=0, step=0,
                  refresh=False):
    """EF + differential quantisation against the history ref.  Returns
    (codes, scales, err' or None, ref')."""
    g = _f32(grad)
    e = _f32(err) if err is not None else None
    r = _f32(ref)
    n = g.size
    m = _mode(mode)
    cb = codes_bytes(n, bits, m)
    sf = scales_floats(n, group, m)
    codes = np.zeros(max(cb, 1), dtype=np.uint8)
    scales = np.zeros(max(sf, 1), dtype=np.float32)
    _check(lib().orc_ef_diff_quant(_p(g, _f32p), _p(e, _f32p) if e is not None else None,
                                   _p(r, _f32p), n, bits, group, m, _rounding(rounding), seed,
                                   step, 1 if refresh else 0, _p(codes, _u8p),
                                   _p(scales, _f32p)), "orc_ef_diff_quant")
    return codes[:cb], scales[:sf], e, r


def diff_dequant(codes, scales, ref, n, bits, group, mode, refresh=False):
    """The receiving side of differential quantisation: returns ref'."""
    c = np.ascontiguousarray(codes, dtype=np.uint8).copy()
    s = _f32(scales)
    r = _f32(ref)
    if c.size == 0:
        c = np.zeros(1, dtype=np.uint8)
    if s.size == 0:
        s = np.zeros(1, dtype=np.float32)
    _check(lib().orc_diff_dequant(_p(c, _u8p), _p(s, _f32p), n, bits, group, _mode(mode),
                                  1 if refresh else 0, _p(r, _f32p)), "orc_diff_dequant")
    return r


def ef_topk_quant(grad, err, k, bits, group, rounding="nearest_even", seed=0,
                  step=0):
    """EF + Top-K + QSGD on the kept values.

    Returns (idx int32[k], codes, scales, err')."""
    g = _f32(grad)
    e = _f32(err)
    n = g.size
    cb = codes_bytes(k, bits, QSGD)
    sf = scales_floats(k, group, QSGD)
    idx = np.zeros(max(k, 1), dtype=np.int32)
    codes = np.zeros(max(cb, 1), dtype=np.uint8)
    scales = np.zeros(max(sf, 1), dtype=np.float32)
    _check(lib().orc_ef_topk_quant(_p(g, _f32p), _p(e, _f32p), n, k, bits,
                                   group, _rounding(rounding), seed, step,
                                   _p(idx, _i32p), _p(codes, _u8p),
                                   _p(scales, _f32p)), "orc_ef_topk_quant")
    return idx[:k], codes[:cb], scales[:sf], e


def ef_randk(grad, err, p, seed=0, step=0):
    """EF + random sparsification: keep i when uniform(seed, step, i) < p.
    Returns (idx int32[kept], val float32[kept], err' or None)."""
    g = _f32(grad)
    n = g.size
    e = _f32(err) if err is not None else None
    idx = np.zeros(max(n, 1), dtype=np.int32)
    val = np.zeros(max(n, 1), dtype=np.float32)
    count = _i64(0)
    _check(lib().orc_ef_randk(_p(g, _f32p), _p(e, _f32p) if e is not None else None, n,
                              float(p), seed, step, _p(idx, _i32p), _p(val, _f32p), n,
                              ctypes.byref(count)), "orc_ef_randk")
    k = count.value
    return idx[:k], val[:k], e


def diagnostics(grad, err, idx, g_hat):
    """(sum c^2, sum g_hat^2, sum e'^2) of one compressed bucket as float64
    [3]: c = grad + err (or grad), g_hat the reconstructed kept values at
    the increasing indices idx, e' = c - g_hat there and c elsewhere."""
    g = _f32(grad)
    e = _f32(err) if err is not None else None
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    gh = _f32(g_hat)
    out = np.zeros(3, dtype=np.float64)
    _check(lib().orc_diagnostics(_p(g, _f32p), _p(e, _f32p) if e is not None else None, g.size,
                                 _p(ix, _i32p), _p(gh, _f32p), ix.size,
                                 out.ctypes.data_as(ctypes.POINTER(ctypes.c_double))),
           "orc_diagnostics")
    return out


def _rank_rows(a, W, k, dtype):
    """(W, k) per-rank rows in the layout the aggregation takes: rank w at
    w * K, K = k rounded up to a multiple of 4 (the padding is zero)."""
    a = np.asarray(a, dtype=dtype).reshape(W, k)
    K = -(-k // 4) * 4
    out = np.zeros((W, K), dtype=dtype)
    out[:, :k] = a
    out = out.reshape(-1)
    return out if out.size else np.zeros(1, dtype)


def topk_aggregate(idx, val, W, k, n):
    """Sum of W ranks' sparse vectors in rank order.  idx, val: (W, k)
    per-rank rows (any shape of W * k entries).  Returns float32[n]."""
    ix = _rank_rows(idx, W, k, np.int32)
    v = _rank_rows(val, W, k, np.float32)
    out = np.zeros(max(n, 1), dtype=np.float32)
    _check(lib().orc_topk_aggregate(W, k, _p(ix, _i32p), _p(v, _f32p), n, _p(out, _f32p)),
           "orc_topk_aggregate")
    return out[:n]


def topk_quant_aggregate(idx, codes, scales, W, k, bits, group, n):
    """Sum of W ranks' QSGD-compressed sparse vectors in rank order; idx as
    (W, k) rows, rank w's codes at w * codes_bytes(k), its scales at
    w * (scales_floats(k) rounded up to a multiple of 4)."""
    ix = _rank_rows(idx, W, k, np.int32)
    c = np.ascontiguousarray(codes, dtype=np.uint8).reshape(-1)
    s = np.ascontiguousarray(scales, dtype=np.float32).reshape(-1)
    sf = -(-scales_floats(k, group, QSGD) // 4) * 4
    if c.size != W * codes_bytes(k, bits, QSGD) or s.size != W * sf:
        raise OracleError("codes / scales do not hold W ranks")
    c = c if c.size else np.zeros(1, np.uint8)
    s = s if s.size else np.zeros(1, np.float32)
    out = np.zeros(max(n, 1), dtype=np.float32)
    _check(lib().orc_topk_quant_aggregate(W, k, _p(ix, _i32p), _p(c, _u8p), _p(s, _f32p),
                                          bits, group, n, _p(out, _f32p)),
           "orc_topk_quant_aggregate")
    return out[:n]


def powersgd_step(grad, err, Q, r):
    """One PowerSGD step on an m x n matrix.  Returns (P_hat, Q', err')."""
    g = _f32(grad)
    if g.ndim != 2:
        raise OracleError("powersgd_step wants a 2-D gradient")
    m, n = g.shape
    e = _f32(err).reshape(m, n)
    q = _f32(Q).reshape(n, r)
    P = np.zeros((m, r), dtype=np.float32)
    _check(lib().orc_powersgd_step(_p(g, _f32p), _p(e, _f32p), m, n, r,
                                   _p(P, _f32p), _p(q, _f32p)),
           "orc_powersgd_step")
    return P, q, e
