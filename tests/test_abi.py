"""The C-ABI library loads and exports every declared symbol; host-side checks.

No GPU is needed: every call here is rejected by argument validation before
any CUDA work, or touches no device state.
"""

import ctypes
import os
import re

import pytest

from domain_backprojection_sarbp_gb300 import _native, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sarbp.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _native.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sarbp_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert sorted(_native.EXPORTS) == declared_functions()


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(6):
        assert lib.sarbp_status_string(code)
    assert lib.sarbp_status_string(99) == b"unknown status"


def _params(**kw):
    base = dict(nx=64, ny=64, na=16, nr=256, x0=-16.0, y0=-16.0, z0=0.0, dx=0.5, dy=0.5,
                r0=8400.0, dr=0.8333, wavelength=0.0312)
    base.update(kw)
    return _native.Params.from_dict(base)


@pytest.mark.parametrize("bad", [
    dict(nx=-1), dict(ny=-3), dict(na=-1), dict(nr=-2), dict(dx=0.0), dict(dy=-0.5),
    dict(dr=0.0), dict(dr=float("nan")), dict(dx=float("inf")), dict(wavelength=0.0),
    dict(wavelength=float("nan")), dict(flags=8), dict(flags=6), dict(nx=1 << 16, ny=1 << 16),
])
def test_plan_rejects_bad_params(lib, bad):
    h = ctypes.c_void_p(123)
    p = _params(**bad)
    assert lib.sarbp_plan(ctypes.byref(h), ctypes.byref(p)) == _native.SARBP_ERR_INVALID_ARG
    assert h.value is None


def test_null_arguments(lib):
    p = _params()
    assert lib.sarbp_plan(None, ctypes.byref(p)) == _native.SARBP_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert lib.sarbp_plan(ctypes.byref(h), None) == _native.SARBP_ERR_INVALID_ARG
    assert lib.sarbp_backproject(None, None, None, None, ctypes.byref(p), None) == \
        _native.SARBP_ERR_INVALID_ARG
    assert lib.sarbp_backproject_host(None, None, None, None, ctypes.byref(p), None) == \
        _native.SARBP_ERR_INVALID_ARG
    assert lib.sarbp_destroy(None) == _native.SARBP_OK
    assert lib.sarbp_last_error(None) == b""
    assert lib.sarbp_plan_describe(None, None) == _native.SARBP_ERR_INVALID_ARG
    assert lib.sarbp_set_timing(None, 1) == _native.SARBP_ERR_INVALID_ARG
    ms, n = ctypes.c_double(), ctypes.c_int32()
    assert lib.sarbp_kernel_times(None, ctypes.byref(ms), ctypes.byref(n)) == \
        _native.SARBP_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_native, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_native, "_lib", None)
    with pytest.raises(ImportError):
        _native.lib()


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "domain_backprojection_sarbp_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f), errors="replace").read()
                assert "oracle" not in text.lower(), f"{f} mentions the oracle"
