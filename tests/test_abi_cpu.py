"""CPU-only checks of the C ABI: the library builds for sm_103a, loads, exports
every entry point that include/trimul.h declares, and rejects bad arguments
before touching a device."""

import ctypes
import os
import re

import pytest

from co_folding_pair_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "trimul.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(trimul_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("trimul_create", "trimul_prepare", "trimul_forward", "trimul_destroy", "trimul_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} is declared in trimul.h but not exported"
        assert name in _lib.SIGNATURES, f"{name} has no ctypes signature"


def test_errors_before_any_device_work(lib):
    p = _lib.TrimulParams()
    h = ctypes.c_void_p()
    assert lib.trimul_create(None, ctypes.byref(p), 0) == 1
    assert lib.trimul_create(ctypes.byref(h), None, 0) == 1
    p.D, p.C, p.eps = 30, 32, 1e-5
    assert lib.trimul_create(ctypes.byref(h), ctypes.byref(p), 0) == 2
    assert "D (30)" in lib.trimul_last_error().decode()
    p.D, p.C = 32, 512
    assert lib.trimul_create(ctypes.byref(h), ctypes.byref(p), 0) == 2
    p.D, p.C, p.eps = 32, 32, 0.0
    assert lib.trimul_create(ctypes.byref(h), ctypes.byref(p), 0) == 1
    p.eps = 1e-5
    assert lib.trimul_create(ctypes.byref(h), ctypes.byref(p), 0) == 1  # null weight pointers
    assert lib.trimul_forward(None, None, None, 1, 8, 0, None, None, 0) == 1
    assert lib.trimul_prepare(None, 1, 8, 1) == 1
    assert lib.trimul_destroy(None) == 0
    assert lib.trimul_kernels_per_forward(None, 1, 64) == -1  # null handle
    assert lib.trimul_kernels_per_forward_host(None, 1, 64) == -1  # null handle
    assert lib.trimul_host_join(None, None) == 1  # null handle
    g = _lib.TrimulGrads()
    assert lib.trimul_backward(None, None, None, None, 1, 8, 0, None, ctypes.byref(g), None, 0) == 1
    assert lib.trimul_backward_workspace_bytes(None, 1, 8) == 0
    assert lib.trimul_kernels_per_backward(None, 1, 8) == -1


def test_product_path_has_no_oracle_import():
    """The package must never reach the CPU oracle."""
    pkg = os.path.dirname(_lib.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(root, f)).read()
                assert "oracle" not in text.replace("oracle/", "").lower() or f == "synthetic.py", f
