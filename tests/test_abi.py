"""The C-ABI library without a GPU: it loads, exports every entry point that
include/hs.h declares, and its host-side argument checks answer before any
CUDA call (so they run on a machine without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def hs():
    from hierarchical_kv_cache_hs_gb300 import build
    build.build_libhs()
    from hierarchical_kv_cache_hs_gb300 import hs as mod
    return mod


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b(hs_[a-z0-9_]+)\s*\(", text):
            names.append(m.group(1))
    return sorted(set(names))


def test_exports_every_declared_symbol(hs):
    names = _declared_functions()
    assert "hs_create" in names and "hs_resolve" in names and "hs_stats" in names
    lib = ctypes.CDLL(hs.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_error_strings(hs):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert hs.hs_error_string(code) != "unknown error"
    assert hs.hs_error_string(-99) == "unknown error"


@pytest.mark.parametrize("args,code", [
    ((0, 1024, 1152, 64, 16, 0), -1),        # no requests
    ((4, 0, 1152, 64, 16, 0), -1),           # empty context
    ((4, 1024, 1000, 64, 16, 0), -1),        # row bytes not a multiple of 16
    ((4, 1024, 1152, 0, 16, 0), -1),         # no slots
    ((4, 1024, 1152, 64, 0, 0), -1),         # no host pool
    ((4, 1024, 1152, 64, 16, -1), -1),       # negative tail
    ((4, 1024, 1152, 64, 16, 2048), -1),     # tail longer than the context
    ((4, 1024, 1152, 64, 15, 0), -3),        # 15 * 64 host rows < 1024 cold tokens
    ((5000, 1024, 1152, 64, 16, 0), -6),     # batch beyond the limit
    ((4, 1024, 1152, 20000, 1, 0), -6),      # slots beyond the limit
    ((4, 1024, 1 << 17, 64, 16, 0), -6),     # row beyond the limit
])
def test_create_argument_checks(hs, args, code):
    rc, h = hs.hs_create_rc(*args)
    assert rc == code and not h


def test_null_handle_is_rejected(hs):
    assert hs.hs_resolve_rc(None, 1, 4, 1) == hs.HS_ERR_ARG
    assert hs.lib.hs_stats(None, None, None) == hs.HS_ERR_ARG
    assert hs.lib.hs_reset(None) == hs.HS_ERR_ARG
    assert hs.hs_host_pool(None) == 0
    assert hs.lib.hs_append(None, None, None) == hs.HS_ERR_ARG
    assert hs.lib.hs_h2d_read(None, None, 16, 0, None) == hs.HS_ERR_ARG
    assert hs.lib.hs_h2d_read(1, 1, 15, 0, None) == hs.HS_ERR_ARG
    assert hs.lib.hs_reset_requests(None, None, 0, None, None) == hs.HS_ERR_ARG
    assert hs.lib.hs_resolve_layers_host(None, 1, None, 4, None, None) == hs.HS_ERR_ARG
    hs.hs_destroy(None)  # no-op


def test_resolve_layers_host_checks(hs):
    rc = hs.hs_resolve_layers_rc
    assert rc([], [], 4, []) == hs.HS_ERR_ARG
    assert rc([None], [1], 4, [1]) == hs.HS_ERR_ARG
    assert rc([1], [1], 0, [1]) == hs.HS_ERR_ARG
    n = hs.HS_MAX_LAYERS + 1
    assert rc([1] * n, [1] * n, 4, [1] * n) == hs.HS_ERR_LIMIT
    assert hs.lib.hs_resolve_layers(None, 1, None, 4, None, None) == hs.HS_ERR_ARG
