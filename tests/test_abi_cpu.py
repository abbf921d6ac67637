"""The C ABI library without a GPU: it loads, exports every entry point that include/pkv.h declares,
and its host-only functions and host-side argument checks behave as documented (no compute call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_decode_pkv_gb300 import _build

    if _build.stale():
        _build.build()
    import paged_kv_decode_pkv_gb300 as pkv

    return pkv.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ["pkv_create_cache", "pkv_append_rope", "pkv_decode_attention", "pkv_combine", "pkv_destroy",
                     "pkv_check_status", "pkv_status_string", "pkv_plan_decode", "pkv_partial_bytes",
                     "pkv_rope_table_bytes", "pkv_pool_bytes"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libpkv.so does not export {name}"


def test_host_only_functions(lib):
    import paged_kv_decode_pkv_gb300 as pkv

    assert pkv.pool_bytes(10, 8, 128) == 10 * 2 * 8 * 16 * 128 * 2
    assert pkv.rope_table_bytes(100, 64) == 100 * 32 * 2 * 4
    assert pkv.partial_bytes(2, 4, 3, 96) == 2 * 4 * 3 * 96 * 4
    assert pkv.pool_bytes(0, 8, 128) == 0
    assert pkv.status_string(pkv.OK) == "ok"
    for code in range(6):
        assert pkv.status_string(code)


def test_argument_errors_return_before_any_device_work(lib):
    import paged_kv_decode_pkv_gb300 as pkv

    P = ctypes.c_void_p
    assert lib.pkv_create_cache(None, None) == pkv.ERR_INVALID_ARG
    out = ctypes.c_void_p()
    d = pkv._Desc(1, 10, 16, 8, 3, 128, 100, 1e4, None, None, None, 0)
    assert lib.pkv_create_cache(ctypes.byref(d), ctypes.byref(out)) == pkv.ERR_INVALID_ARG
    assert lib.pkv_append_rope(None, 0, None, None, None, None, None, 1, 1, None, None, None, None) == \
        pkv.ERR_INVALID_ARG
    used = ctypes.c_int()
    assert lib.pkv_decode_attention(None, 0, None, None, None, None, None, 1, 1, 0, 0, 0, 4, 0.0, None, None,
                                    ctypes.byref(used), None) == pkv.ERR_INVALID_ARG
    assert lib.pkv_combine(None, None, None, None, 1, 4, 2, 100, None, None, None) == pkv.ERR_UNSUPPORTED
    assert lib.pkv_combine(None, None, None, None, 1, 4, 0, 128, None, None, None) == pkv.ERR_INVALID_ARG
    assert lib.pkv_combine(None, None, None, None, 0, 4, 2, 128, None, None, None) == pkv.OK
    assert lib.pkv_check_status(None, None, None) == pkv.ERR_INVALID_ARG
    assert lib.pkv_set_wait_limit(None, 1) == pkv.ERR_INVALID_ARG
    assert lib.pkv_set_stage_stall(None, 1) == pkv.ERR_INVALID_ARG
    s, c = ctypes.c_int(), ctypes.c_int()
    assert lib.pkv_plan_decode(None, 1, 1, 0, 0, 0, 4, ctypes.byref(s), ctypes.byref(c)) == pkv.ERR_INVALID_ARG
    assert lib.pkv_device_info(None, 8, ctypes.byref(s), ctypes.byref(c)) == pkv.ERR_INVALID_ARG
    lib.pkv_destroy(None)


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    import paged_kv_decode_pkv_gb300 as pkv

    monkeypatch.setattr(pkv, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(pkv, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        pkv.lib()


def test_int8_cache_takes_one_query_head_per_kv_head(lib):
    """The int8 cache runs on the tensor-core path for every group size: a cache with one query
    head per KV head passes the argument checks (without a GPU it then fails at the device step)."""
    import ctypes

    import paged_kv_decode_pkv_gb300 as pkv

    pools = (ctypes.c_void_p * 1)(256)
    d = pkv._Desc(1, 10, 16, 8, 8, 128, 100, 1e4, ctypes.cast(pools, ctypes.POINTER(ctypes.c_void_p)), 256, 256,
                  pkv.OPT_INT8_KV)
    out = ctypes.c_void_p()
    assert lib.pkv_create_cache(ctypes.byref(d), ctypes.byref(out)) == pkv.ERR_CUDA
    assert lib.pkv_pool_bytes_int8(10, 8, 128) == 10 * 2 * 8 * (16 * 128 + 64)
