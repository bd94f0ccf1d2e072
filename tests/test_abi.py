"""The C-ABI library builds for sm_103a, loads, exports every declared symbol,
and validates arguments on the host (no GPU needed for any of this)."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "moe_w4a16.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_w4a16_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import int4_weight_only_moe_gb300 as pkg
    return pkg.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moe_w4a16_create", "moe_w4a16_pack", "moe_w4a16_forward",
                     "moe_w4a16_workspace_size", "moe_w4a16_destroy", "moe_w4a16_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_wraps_every_symbol():
    import int4_weight_only_moe_gb300 as pkg
    for name in declared_functions():
        assert callable(getattr(pkg, name)), name


def test_create_rejects_bad_shapes_without_touching_the_gpu(lib):
    h = ctypes.c_void_p()
    cases = [(8, 256, 128, 2, 16), (8, 200, 128, 2, 32), (8, 256, 96, 2, 32), (8, 256, 192, 2, 32),
             (0, 256, 128, 2, 32), (8, 256, 128, 9, 32), (2000, 256, 128, 2, 32)]
    for E, K, N, k, g in cases:
        rc = lib.moe_w4a16_create(E, K, N, k, g, ctypes.byref(h))
        assert rc == -2, (E, K, N, k, g)
        assert lib.moe_w4a16_last_error()
    assert lib.moe_w4a16_create(8, 256, 128, 2, 32, None) == -1


def test_null_handle_paths(lib):
    assert lib.moe_w4a16_workspace_size(None, 4) == 0
    assert lib.moe_w4a16_packed_bytes(None) == 0
    assert lib.moe_w4a16_destroy(None) == -1
    assert lib.moe_w4a16_set_option(None, 1, 4) == -1
    assert b"null" in lib.moe_w4a16_last_error()


def test_align_debug_rejects_bad_arguments(lib):
    buf = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    assert lib.moe_w4a16_align_debug(buf, 4, 0, 8, 16, buf, buf, buf, 1000, None) == -1
    assert lib.moe_w4a16_align_debug(buf, 4, 2, 8, 16, buf, buf, buf, 8, None) == -1
    assert lib.moe_w4a16_align_debug(buf, 4, 2, 2000, 16, buf, buf, buf, 1000, None) == -1


def test_package_fails_loudly_without_library(monkeypatch):
    import int4_weight_only_moe_gb300 as pkg
    monkeypatch.setattr(pkg, "_LIB", None)
    monkeypatch.setattr(pkg, "LIB_PATH", "/nonexistent/libmoe_w4a16.so")
    with pytest.raises(RuntimeError):
        pkg.lib()
