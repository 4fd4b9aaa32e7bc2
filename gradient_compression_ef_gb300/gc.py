"""ctypes binding of ``libgc.so`` (the C ABI declared in include/gc.h).

Argument marshalling only: every step of the compressor runs in the CUDA
kernels of the library.  Functions take torch CUDA tensors (or raw device
addresses as ints) and pass ``data_ptr()`` values through unchanged.  There
is no fallback: importing this module raises if the library is missing.

    from gradient_compression_ef_gb300 import gc
    ctx = gc.Context(max_n)                  # bound to the current stream
    gc.ef_topk(ctx, grad, err, k, idx, val)  # asynchronous on ctx's stream
    ctx.check()                              # sync + device status
"""
import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libgc.so")

MINMAX, QSGD, TERN, LOG = 0, 1, 2, 3
NEAREST_EVEN, STOCHASTIC = 0, 1
MODES = {"minmax": MINMAX, "qsgd": QSGD, "tern": TERN, "log": LOG}
ROUNDINGS = {"nearest_even": NEAREST_EVEN, "stochastic": STOCHASTIC}

PHASE_COUNT = 25

OK = 0
ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIGNMENT, ERR_WORKSPACE = -1, -2, -3, -4
ERR_CUDA, ERR_DEVICE_CHECK, ERR_NO_MEMORY = -5, -6, -7

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64
_int = ctypes.c_int

# (name, restype, argtypes) of every function declared in include/gc.h
SIGNATURES = [
    ("gc_version", _int, []),
    ("gc_status_string", ctypes.c_char_p, [_int]),
    ("gc_ctx_create", _int, [ctypes.POINTER(_vp), _vp, _i64]),
    ("gc_ctx_destroy", _int, [_vp]),
    ("gc_ctx_set_stream", _int, [_vp, _vp]),
    ("gc_ctx_reserve_powersgd", _int, [_vp, _i64, _i64, _int]),
    ("gc_ctx_check", _int, [_vp]),
    ("gc_phase_name", ctypes.c_char_p, [_int]),
    ("gc_ctx_enable_timing", _int, [_vp, _int]),
    ("gc_ctx_read_timing", _int, [_vp, ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_int64)]),
    ("gc_ctx_launch_count", _i64, [_vp]),
    ("gc_codes_bytes", _i64, [_i64, _int, _int]),
    ("gc_scales_floats", _i64, [_i64, _i64, _int]),
    ("gc_ef_topk", _int, [_vp, _vp, _vp, _i64, _i64, _vp, _vp]),
    ("gc_quant", _int, [_vp, _vp, _i64, _int, _i64, _int, _int, _u64, _u64, _vp, _vp]),
    ("gc_dequant", _int, [_vp, _vp, _vp, _i64, _int, _i64, _int, _vp]),
    ("gc_ef_quant", _int, [_vp, _vp, _vp, _i64, _int, _i64, _int, _int, _u64, _u64, _vp, _vp]),
    ("gc_ef_topk_quant", _int, [_vp, _vp, _vp, _i64, _i64, _int, _i64, _int, _u64, _u64,
                                _vp, _vp, _vp]),
    ("gc_ef_diff_quant", _int, [_vp, _vp, _vp, _vp, _i64, _int, _i64, _int, _int, _u64, _u64,
                                _int, _vp, _vp]),
    ("gc_diff_dequant", _int, [_vp, _vp, _vp, _i64, _int, _i64, _int, _int, _vp]),
    ("gc_powersgd_step", _int, [_vp, _vp, _vp, _i64, _i64, _int, _vp, _vp]),
    ("gc_ef_topk_noalloc", _int, [_vp, _vp, _i64, _i64, _vp, _vp, _vp]),
    ("gc_bucket_seed", _u64, [_u64, _int]),
    ("gc_ctx_set_buckets", _int, [_vp, _int, ctypes.POINTER(_i64), ctypes.POINTER(_i64)]),
    ("gc_ctx_set_deferred_residual", _int, [_vp, _int]),
    ("gc_bucket_flush", _int, [_vp]),
    ("gc_bucket_offsets", _int, [_int, ctypes.POINTER(_i64), _int, _i64, ctypes.POINTER(_i64),
                                 ctypes.POINTER(_i64), ctypes.POINTER(_i64)]),
    ("gc_ef_topk_buckets", _int, [_vp, _vp, _vp, _vp, _vp, _vp]),
    ("gc_ef_topk_quant_buckets", _int, [_vp, _vp, _vp, _int, _i64, _int, _u64, _u64, _vp, _vp,
                                        _vp, _vp]),
    ("gc_ef_randk", _int, [_vp, _vp, _vp, _i64, ctypes.c_float, _u64, _u64, _vp, _vp, _i64,
                           _vp]),
    ("gc_topk_aggregate", _int, [_vp, _int, _i64, _vp, _vp, _i64, _vp]),
    ("gc_topk_quant_aggregate", _int, [_vp, _int, _i64, _vp, _vp, _vp, _int, _i64, _i64, _vp]),
]

# largest n of gc_ef_topk_noalloc (GC_NOALLOC_MAX_N in include/gc.h)
NOALLOC_MAX_N = 1048576


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            "libgc.so is not built (%s); run `python -c \"import __graft_entry__ as g; "
            "g.build()\"` first -- there is no non-CUDA fallback" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class GCError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s: %s (%d)" % (what, status_string(status), status))


def phase_name(phase):
    return lib.gc_phase_name(phase).decode()


def status_string(status):
    return lib.gc_status_string(status).decode()


def _check(status, what):
    if status != OK:
        raise GCError(status, what)


def _ptr(t):
    """Device address of a tensor (or an int address / None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _mode(m):
    return MODES[m] if isinstance(m, str) else int(m)


def _rounding(r):
    return ROUNDINGS[r] if isinstance(r, str) else int(r)


def codes_bytes(n, bits, mode):
    return int(lib.gc_codes_bytes(n, bits, _mode(mode)))


def scales_floats(n, group, mode):
    return int(lib.gc_scales_floats(n, group, _mode(mode)))


class Context:
    """A gc_ctx: scratch for calls of up to ``max_n`` elements, bound to a
    CUDA stream (default: torch's current stream at creation)."""

    def __init__(self, max_n, stream=None):
        if stream is None:
            import torch
            stream = torch.cuda.current_stream()
        handle = stream if isinstance(stream, int) else stream.cuda_stream
        self._stream_ref = stream
        h = _vp()
        _check(lib.gc_ctx_create(ctypes.byref(h), handle, max_n), "gc_ctx_create")
        self.handle = h
        self.max_n = max_n

    def set_stream(self, stream):
        handle = stream if isinstance(stream, int) else stream.cuda_stream
        _check(lib.gc_ctx_set_stream(self.handle, handle), "gc_ctx_set_stream")
        self._stream_ref = stream

    def reserve_powersgd(self, max_m, max_n, max_r):
        _check(lib.gc_ctx_reserve_powersgd(self.handle, max_m, max_n, max_r),
               "gc_ctx_reserve_powersgd")

    def check(self):
        _check(lib.gc_ctx_check(self.handle), "gc_ctx_check")

    def enable_timing(self, max_launches):
        """Brackets each later kernel launch with CUDA events on the stream."""
        _check(lib.gc_ctx_enable_timing(self.handle, max_launches), "gc_ctx_enable_timing")

    def read_timing(self):
        """{phase name: (total ms, launches)} of the timed launches since the
        last read (synchronises the stream)."""
        ms = (ctypes.c_double * PHASE_COUNT)()
        cnt = (ctypes.c_int64 * PHASE_COUNT)()
        _check(lib.gc_ctx_read_timing(self.handle, ms, cnt), "gc_ctx_read_timing")
        return {phase_name(p): (ms[p], cnt[p]) for p in range(PHASE_COUNT) if cnt[p]}

    def launch_count(self):
        return int(lib.gc_ctx_launch_count(self.handle))

    def set_buckets(self, bucket_n, bucket_k):
        """Bucket plan: consecutive slices of bucket_n[b] elements keeping
        bucket_k[b] entries each (synchronous)."""
        nb = len(bucket_n)
        if len(bucket_k) != nb:
            raise ValueError("bucket_n and bucket_k differ in length")
        an = (_i64 * max(nb, 1))(*[int(v) for v in bucket_n])
        ak = (_i64 * max(nb, 1))(*[int(v) for v in bucket_k])
        _check(lib.gc_ctx_set_buckets(self.handle, nb, an, ak), "gc_ctx_set_buckets")
        self.bucket_n = [int(v) for v in bucket_n]
        self.bucket_k = [int(v) for v in bucket_k]

    def set_deferred_residual(self, on):
        """on: the bucketed calls with error feedback keep the kept entries'
        residuals aside and the next bucketed call on the same err applies
        them as it reads e; err is exact only after bucket_flush().  off:
        flushes, then writes e' in full again."""
        _check(lib.gc_ctx_set_deferred_residual(self.handle, 1 if on else 0),
               "gc_ctx_set_deferred_residual")

    def bucket_flush(self):
        """Writes the pending residuals of the last deferred bucketed call into
        its err (asynchronous on the context's stream)."""
        _check(lib.gc_bucket_flush(self.handle), "gc_bucket_flush")

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            st = lib.gc_ctx_destroy(self.handle)
            self.handle = None
            _check(st, "gc_ctx_destroy")

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            if getattr(self, "handle", None) is not None and self.handle.value:
                lib.gc_ctx_destroy(self.handle)
        except Exception:
            pass


def ef_topk(ctx, grad, err, k, idx_out, val_out, n=None):
    n = grad.numel() if n is None else n
    _check(lib.gc_ef_topk(ctx.handle, _ptr(grad), _ptr(err), n, k, _ptr(idx_out),
                          _ptr(val_out)), "gc_ef_topk")


def quant(ctx, x, bits, group, mode, rounding, seed, step, codes_out, scales_out, n=None):
    n = x.numel() if n is None else n
    _check(lib.gc_quant(ctx.handle, _ptr(x), n, bits, group, _mode(mode), _rounding(rounding),
                        seed, step, _ptr(codes_out), _ptr(scales_out)), "gc_quant")


def dequant(ctx, codes, scales, n, bits, group, mode, x_out):
    _check(lib.gc_dequant(ctx.handle, _ptr(codes), _ptr(scales), n, bits, group, _mode(mode),
                          _ptr(x_out)), "gc_dequant")


def ef_quant(ctx, grad, err, bits, group, mode, rounding, seed, step, codes_out, scales_out,
             n=None):
    n = grad.numel() if n is None else n
    _check(lib.gc_ef_quant(ctx.handle, _ptr(grad), _ptr(err), n, bits, group, _mode(mode),
                           _rounding(rounding), seed, step, _ptr(codes_out),
                           _ptr(scales_out)), "gc_ef_quant")


def ef_diff_quant(ctx, grad, err, ref, bits, group, mode, rounding, seed, step, refresh,
                  codes_out, scales_out, n=None):
    """Differential quantisation against the history ref (updated in place);
    err may be None."""
    n = grad.numel() if n is None else n
    _check(lib.gc_ef_diff_quant(ctx.handle, _ptr(grad), _ptr(err), _ptr(ref), n, bits, group,
                                _mode(mode), _rounding(rounding), seed, step,
                                1 if refresh else 0, _ptr(codes_out), _ptr(scales_out)),
           "gc_ef_diff_quant")


def diff_dequant(ctx, codes, scales, n, bits, group, mode, refresh, ref):
    _check(lib.gc_diff_dequant(ctx.handle, _ptr(codes), _ptr(scales), n, bits, group,
                               _mode(mode), 1 if refresh else 0, _ptr(ref)), "gc_diff_dequant")


def ef_topk_quant(ctx, grad, err, k, bits, group, rounding, seed, step, idx_out, codes_out,
                  scales_out, n=None):
    n = grad.numel() if n is None else n
    _check(lib.gc_ef_topk_quant(ctx.handle, _ptr(grad), _ptr(err), n, k, bits, group,
                                _rounding(rounding), seed, step, _ptr(idx_out),
                                _ptr(codes_out), _ptr(scales_out)), "gc_ef_topk_quant")


def powersgd_step(ctx, grad, err, m, n, r, P_out, Q_inout):
    _check(lib.gc_powersgd_step(ctx.handle, _ptr(grad), _ptr(err), m, n, r, _ptr(P_out),
                                _ptr(Q_inout)), "gc_powersgd_step")


def ef_topk_noalloc(grad, err, k, idx_out, val_out, stream=None, n=None):
    """gc_ef_topk_noalloc: EF + Top-K with no context and no allocation, on
    ``stream`` (default: torch's current stream); n <= NOALLOC_MAX_N."""
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    handle = stream if isinstance(stream, int) else stream.cuda_stream
    n = grad.numel() if n is None else n
    _check(lib.gc_ef_topk_noalloc(_ptr(grad), _ptr(err), n, k, _ptr(idx_out), _ptr(val_out),
                                  handle), "gc_ef_topk_noalloc")


def bucket_seed(seed, b):
    """The Philox key the bucketed calls give bucket b for ``seed``."""
    return int(lib.gc_bucket_seed(seed, b))


def bucket_offsets(bucket_k, bits=None, group=None):
    """gc_bucket_offsets: (idx_off, codes_off, scales_off), each a list of
    nb + 1 starts (the last is the total); codes_off / scales_off are None
    when bits / group are not given."""
    nb = len(bucket_k)
    ak = (_i64 * max(nb, 1))(*[int(v) for v in bucket_k])
    oi = (_i64 * (nb + 1))()
    oc = (_i64 * (nb + 1))() if bits is not None else None
    os_ = (_i64 * (nb + 1))() if group is not None else None
    _check(lib.gc_bucket_offsets(nb, ak, 0 if bits is None else bits,
                                 0 if group is None else group, oi, oc, os_),
           "gc_bucket_offsets")
    return (list(oi), list(oc) if oc is not None else None,
            list(os_) if os_ is not None else None)


def ef_topk_buckets(ctx, grad, err, idx_out, val_out, diag=None):
    """diag: None, or a device float64 tensor of 3 * nb values receiving per
    bucket (sum c^2, sum g_hat^2, sum e'^2)."""
    _check(lib.gc_ef_topk_buckets(ctx.handle, _ptr(grad), _ptr(err), _ptr(idx_out),
                                  _ptr(val_out), _ptr(diag)), "gc_ef_topk_buckets")


def ef_topk_quant_buckets(ctx, grad, err, bits, group, rounding, seed, step, idx_out,
                          codes_out, scales_out, diag=None):
    _check(lib.gc_ef_topk_quant_buckets(ctx.handle, _ptr(grad), _ptr(err), bits, group,
                                        _rounding(rounding), seed, step, _ptr(idx_out),
                                        _ptr(codes_out), _ptr(scales_out), _ptr(diag)),
           "gc_ef_topk_quant_buckets")



def topk_aggregate(ctx, W, k, idx, val, n, out):
    """gc_topk_aggregate: out[n] = rank-ordered sum of W ranks' (idx, val)."""
    _check(lib.gc_topk_aggregate(ctx.handle, W, k, _ptr(idx), _ptr(val), n, _ptr(out)),
           "gc_topk_aggregate")


def topk_quant_aggregate(ctx, W, k, idx, codes, scales, bits, group, n, out):
    """gc_topk_quant_aggregate: the same with QSGD-coded values per rank."""
    _check(lib.gc_topk_quant_aggregate(ctx.handle, W, k, _ptr(idx), _ptr(codes), _ptr(scales),
                                       bits, group, n, _ptr(out)), "gc_topk_quant_aggregate")


def ef_randk(ctx, grad, err, p, seed, step, idx_out, val_out, count_out, n=None, capacity=None):
    """gc_ef_randk: EF + random sparsification; count_out is a device int64
    tensor receiving the kept count."""
    n = grad.numel() if n is None else n
    capacity = idx_out.numel() if capacity is None else capacity
    _check(lib.gc_ef_randk(ctx.handle, _ptr(grad), _ptr(err), n, float(p), seed, step,
                           _ptr(idx_out), _ptr(val_out), capacity, _ptr(count_out)),
           "gc_ef_randk")
