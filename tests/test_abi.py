"""The C ABI without a GPU: the library loads, exports every function the
header declares, and rejects bad limits before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "fdl.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(fdl_[a-z0-9_]+)\s*\(", text)
    return sorted(set(n for n in names if not n.startswith("fdl_KIND")))


@pytest.fixture(scope="module")
def lib():
    from kv_cache_attention_gb300 import build
    import kv_cache_attention_gb300 as fdl
    build.build()
    return fdl.load_library()


def test_header_and_binding_agree():
    import kv_cache_attention_gb300 as fdl
    assert header_functions() == sorted(fdl.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_create_rejects_bad_limits_without_touching_the_device(lib):
    import kv_cache_attention_gb300 as fdl
    good = dict(d_model=256, n_heads=4, head_dim=64, rope_theta=1e4, max_batch=1, max_seq=112,
                max_views=16, page_size=128, n_pages=1, max_rows=112, vocab=1024, dtype="f32")
    for bad in (dict(d_model=255), dict(head_dim=96, d_model=384), dict(max_views=3), dict(page_size=0),
                dict(rope_theta=0.5), dict(vocab=0), dict(max_rows=0)):
        with pytest.raises(fdl.FdlError) as ei:
            fdl.fdl_create(**{**good, **bad}, stream=0)
        assert ei.value.status == fdl.FDL_ERR_INVALID_ARG


def test_null_context_is_rejected(lib):
    import kv_cache_attention_gb300 as fdl
    assert lib.fdl_sync_status(None) == fdl.FDL_ERR_INVALID_ARG
    assert lib.fdl_tile_m(None) == 0
    assert lib.fdl_qkv_rope_cache_write(None, None, None, 0, None, None, None, None, 0, None, None, None) \
        == fdl.FDL_ERR_INVALID_ARG
