"""The C-ABI library: it loads, exports every function include/gc.h declares,
and its host-only calls (sizes, status strings, argument validation) behave
as documented.  No kernel runs here, so these tests need no GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gc.h")


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"GC_API\s+[\w\s\*]+?\b(gc_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def gc():
    import __graft_entry__
    __graft_entry__.build()
    from gradient_compression_ef_gb300 import gc as binding
    return binding


def test_header_declares_the_boundary():
    names = _declared()
    for need in ("gc_ef_topk", "gc_quant", "gc_dequant", "gc_ef_quant", "gc_ef_topk_quant",
                 "gc_powersgd_step", "gc_ctx_create", "gc_ctx_destroy", "gc_codes_bytes",
                 "gc_scales_floats", "gc_status_string"):
        assert need in names


def test_library_exports_every_declared_symbol(gc):
    lib = ctypes.CDLL(gc.LIB_PATH)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    bound = {name for name, _, _ in gc.SIGNATURES}
    assert bound == set(_declared())


def test_sizes_agree_with_the_oracle(gc):
    import oracle
    for n in (0, 1, 5, 63, 64, 65, 1000, 12345, 1 << 20):
        for bits in (1, 2, 4, 8):
            for mode in ("minmax", "qsgd"):
                assert gc.codes_bytes(n, bits, mode) == oracle.codes_bytes(n, bits, mode)
        assert gc.codes_bytes(n, 2, "tern") == oracle.codes_bytes(n, 2, "tern")
        for group in (0, 1, 3, 64, 100, 4096):
            for mode in ("minmax", "qsgd", "tern"):
                assert gc.scales_floats(n, group, mode) == oracle.scales_floats(n, group, mode)
    assert gc.codes_bytes(10, 3, "minmax") == -1
    assert gc.scales_floats(10, -1, "qsgd") == -1


def test_status_strings(gc):
    for st in range(-7, 1):
        assert gc.status_string(st) not in ("", "unknown status")
    assert gc.status_string(-99) == "unknown status"


def test_validation_before_any_device_work(gc):
    """Calls with a NULL context or bad sizes fail on the host."""
    L = gc.lib
    assert L.gc_ef_topk(None, None, None, 10, 1, None, None) == gc.ERR_INVALID_ARG
    assert L.gc_quant(None, None, 10, 8, 64, 0, 0, 0, 0, None, None) == gc.ERR_INVALID_ARG
    assert L.gc_dequant(None, None, None, 10, 8, 64, 0, None) == gc.ERR_INVALID_ARG
    assert L.gc_ef_quant(None, None, None, 10, 8, 64, 0, 0, 0, 0, None, None) == \
        gc.ERR_INVALID_ARG
    assert L.gc_ef_topk_quant(None, None, None, 10, 1, 8, 64, 0, 0, 0, None, None, None) == \
        gc.ERR_INVALID_ARG
    assert L.gc_powersgd_step(None, None, None, 4, 4, 2, None, None) == gc.ERR_INVALID_ARG
    assert L.gc_ctx_create(None, None, 10) == gc.ERR_INVALID_ARG
    assert L.gc_ctx_destroy(None) == gc.OK
    assert L.gc_ctx_check(None) == gc.ERR_INVALID_ARG


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    """With libgc.so absent the binding raises instead of falling back."""
    import importlib.util
    src = os.path.join(ROOT, "gradient_compression_ef_gb300", "gc.py")
    pkg = tmp_path / "fakepkg"
    pkg.mkdir()
    (pkg / "gc.py").write_text(open(src).read())
    spec = importlib.util.spec_from_file_location("fake_gc", str(pkg / "gc.py"))
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)


def test_bucket_offsets_agree_with_the_oracle_sizes(gc):
    """gc_bucket_offsets is the running sum of the per-bucket output sizes
    (indices rounded up to 4 slots, codes as gc_codes_bytes, scales rounded
    up to 4 floats)."""
    import oracle
    ks = [0, 1, 5, 63, 64, 65, 1000, 12345, 65536]
    for bits in (1, 2, 4, 8):
        for group in (4, 64, 128):
            oi, oc, os_ = gc.bucket_offsets(ks, bits, group)
            assert len(oi) == len(oc) == len(os_) == len(ks) + 1
            assert oi[0] == oc[0] == os_[0] == 0
            for b, k in enumerate(ks):
                assert oi[b + 1] - oi[b] == -(-k // 4) * 4
                assert oc[b + 1] - oc[b] == oracle.codes_bytes(k, bits, "qsgd")
                assert os_[b + 1] - os_[b] == -(-oracle.scales_floats(k, group, "qsgd") // 4) * 4
                assert oc[b] % 16 == 0 and (4 * oi[b]) % 16 == 0 and (4 * os_[b]) % 16 == 0
    oi, oc, os_ = gc.bucket_offsets(ks)
    assert oc is None and os_ is None and oi[-1] == sum(-(-k // 4) * 4 for k in ks)


def test_bucket_calls_validate_on_the_host(gc):
    L = gc.lib
    n = (ctypes.c_int64 * 2)(8, 8)
    k = (ctypes.c_int64 * 2)(1, 1)
    assert L.gc_ctx_set_buckets(None, 2, n, k) == gc.ERR_INVALID_ARG
    assert L.gc_ef_topk_buckets(None, None, None, None, None, None) == gc.ERR_INVALID_ARG
    assert L.gc_ef_topk_quant_buckets(None, None, None, 8, 64, 0, 0, 0, None, None, None,
                                      None) == gc.ERR_INVALID_ARG
    out = (ctypes.c_int64 * 3)()
    assert L.gc_bucket_offsets(0, k, 8, 64, out, None, None) == gc.ERR_INVALID_ARG
    assert L.gc_bucket_offsets(2, None, 8, 64, out, None, None) == gc.ERR_INVALID_ARG
    assert L.gc_bucket_offsets(2, k, 3, 64, out, out, None) == gc.ERR_UNSUPPORTED
    bad = (ctypes.c_int64 * 2)(1, -1)
    assert L.gc_bucket_offsets(2, bad, 8, 64, out, None, None) == gc.ERR_INVALID_ARG
    assert L.gc_ctx_set_deferred_residual(None, 1) == gc.ERR_INVALID_ARG
    assert L.gc_ctx_set_deferred_residual(None, 0) == gc.ERR_INVALID_ARG
    assert L.gc_bucket_flush(None) == gc.ERR_INVALID_ARG


def test_bucket_seed_matches_the_oracle(gc):
    import oracle
    for seed in (0, 1, 1000, 0xFFFFFFFFFFFFFFFF, 0x123456789ABCDEF0):
        for b in (0, 1, 2, 20, 255, 65535):
            assert gc.bucket_seed(seed, b) == oracle.bucket_seed(seed, b)
