"""The C-ABI library loads and exports every symbol its header declares (no GPU needed)."""
import ctypes

import pytest

from seismic_wave_propagation_gb300 import _lib
from seismic_wave_propagation_gb300 import build as b


@pytest.fixture(scope="module")
def lib():
    b.build()
    return _lib.load()


def test_exports_every_declared_symbol(lib):
    names = _lib.header_functions()
    assert {"stencil_plan_create", "stencil_apply", "wave_step", "stencil_plan_status",
            "stencil_last_error", "stencil_plan_destroy"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name


def test_host_side_validation_without_device(lib):
    assert lib.stencil_version().decode().startswith("libstencil")
    c = (ctypes.c_float * 6)(*[1.0] * 6)
    assert not lib.stencil_plan_create(64, 64, 64, 0, c)
    assert b"radius" in lib.stencil_last_error()
    assert not lib.stencil_plan_create(64, 64, 64, 5, c)
    assert not lib.stencil_plan_create(62, 64, 64, 1, c)
    assert b"multiple of 4" in lib.stencil_last_error()
    assert not lib.stencil_plan_create(64, 64, 64, 1, None)
    assert lib.stencil_apply(None, None, None, None) == -1
    assert lib.wave_step(None, None, None, None, None, None, None) == -1
    assert lib.stencil_plan_status(None, None) == -1
    lib.stencil_plan_destroy(None)


def test_product_path_has_no_oracle_dependency():
    import pathlib
    root = pathlib.Path(__file__).resolve().parents[1] / "seismic_wave_propagation_gb300"
    for p in list(root.rglob("*.py")) + list(root.rglob("*.cu")) + list(root.rglob("*.cuh")) + list(root.rglob("*.h")):
        text = p.read_text()
        assert "import oracle" not in text and "from oracle" not in text and "stencil_oracle" not in text, p
