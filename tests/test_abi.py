"""The C-ABI library loads and exports every symbol include/moe_reader.h
declares (no GPU, no compute calls)."""

import ctypes
import os
import re

import pytest

from calibration_free_sparse_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe_reader.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_reader_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    path = B.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moe_reader_prepare", "moe_reader_decode", "moe_reader_destroy"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_the_header():
    from calibration_free_sparse_gb300 import reader

    assert sorted(reader.EXPORTED_SYMBOLS) == declared_functions()


def test_host_only_calls(lib):
    lib.moe_reader_abi_version.restype = ctypes.c_int
    assert lib.moe_reader_abi_version() == 1
    lib.moe_reader_strerror.restype = ctypes.c_char_p
    lib.moe_reader_strerror.argtypes = [ctypes.c_int]
    assert b"invalid" in lib.moe_reader_strerror(-1)
    # null handle / null config are rejected without touching a device
    lib.moe_reader_prepare.restype = ctypes.c_int
    out = ctypes.c_void_p()
    assert lib.moe_reader_prepare(None, None, None, None, None, None, ctypes.byref(out)) == -1
    lib.moe_reader_decode.restype = ctypes.c_int
    assert lib.moe_reader_decode(None, None, 1, None, None, 1, None, None) == -1
    lib.moe_reader_destroy(None)


def test_binding_refuses_to_run_without_library(monkeypatch, tmp_path):
    from calibration_free_sparse_gb300 import reader

    monkeypatch.setattr(reader, "_LIB", None)
    monkeypatch.setattr(reader, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        reader.library()
