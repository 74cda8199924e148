"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol include/fnospec.h declares, and rejects bad shapes before it
touches the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from fourier_neural_spectral_gb300 import fnospec
    return fnospec.load_library()


def header_symbols():
    text = open(os.path.join(ROOT, "include", "fnospec.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fno_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    from fourier_neural_spectral_gb300 import fnospec
    assert header_symbols() == sorted(fnospec.EXPORTS)


def test_library_exports_every_header_symbol(lib):
    for name in header_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    from fourier_neural_spectral_gb300 import fnospec
    for code in range(7):
        s = lib.fno_status_string(code).decode()
        assert s.startswith("FNO_")
    assert "unknown" in lib.fno_status_string(99).decode()
    assert fnospec.status_string(fnospec.FNO_ERR_WORKSPACE).startswith("FNO_ERR_WORKSPACE")


@pytest.mark.parametrize("shape,code", [
    ((0, 4, 4, 16, 16, 4, 4), 1),     # B = 0
    ((2, 4, 4, 16, 16, 9, 4), 1),     # 2*m1 > H
    ((2, 4, 4, 16, 16, 4, 10), 1),    # m2 > W/2 + 1
    ((2, 4, 4, 16, 16, 0, 4), 1),     # m1 = 0
    ((2, 4, 4, 8192, 16, 4, 4), 2),   # H above 4096
    ((2, 4, 4, 16, 8192, 4, 4), 2),   # W above 4096
    ((2, 4, 4, 1, 16, 0, 4), 1),      # H = 1 (m1 must be >= 1)
])
def test_plan_create_rejects_bad_shapes(lib, shape, code):
    h = ctypes.c_void_p(1234)
    rc = lib.fno_plan_create(ctypes.byref(h), *shape, 0)
    assert rc == code
    assert not h.value


@pytest.mark.parametrize("shape,code", [
    ((0, 4, 4, 64, 8), 1),       # B = 0
    ((2, 0, 4, 64, 8), 1),       # Cin = 0
    ((2, 4, 4, 64, 0), 1),       # no modes
    ((2, 4, 4, 64, 34), 1),      # m > L/2 + 1
    ((2, 4, 4, 15, 9), 1),       # m > L/2 + 1 for odd L
    ((2, 4, 4, 1, 1), 2),        # L = 1
    ((2, 4, 4, 8192, 8), 2),     # L above 4096
])
def test_plan_create_1d_rejects_bad_shapes(lib, shape, code):
    h = ctypes.c_void_p(1234)
    rc = lib.fno_plan_create_1d(ctypes.byref(h), *shape, 0)
    assert rc == code
    assert not h.value


def test_plan_create_rejects_bad_precision(lib):
    h = ctypes.c_void_p()
    assert lib.fno_plan_create(ctypes.byref(h), 2, 4, 4, 16, 16, 4, 4, 7) == 1


def test_null_arguments(lib):
    assert lib.fno_plan_create(None, 2, 4, 4, 16, 16, 4, 4, 0) == 1
    assert lib.fno_plan_workspace_size(None, None) == 1
    assert lib.fno_plan_execute(None, None, None, None, None, 0, None) == 1
    assert lib.fno_plan_destroy(None) == 0
    assert lib.fno_forward_modes(None, None, None, None, 0, None) == 1
    assert lib.fno_mix_modes(None, None, None, None, None) == 1
    assert lib.fno_inverse_modes(None, None, None, None, 0, None) == 1
    assert lib.fno_get_device_status(None, None) == 1


def test_one_shot_rejects_bad_shape_before_device(lib):
    assert lib.fno_spectral_conv2d(None, None, None, 2, 4, 4, 16, 16, 9, 4, None) == 1
