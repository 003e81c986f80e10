"""The debug build of the library (bounds-checked stores, NVTX ranges around every C-ABI
call) compiles for sm_103a and loads without a GPU: every entry point of include/gqa.h is
exported, plus the store guard's probe, and the NVTX hooks are linked in (the product
library has neither)."""
import ctypes
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def debug_lib():
    from sliding_window_gb300 import build
    return build.build(checked=True)


def test_debug_library_loads_and_exports_the_abi(debug_lib):
    from sliding_window_gb300 import gqa
    lib = ctypes.CDLL(debug_lib)
    for name in gqa.EXPORTED + ["gqa_test_bounds_check"]:
        assert hasattr(lib, name), name
    lib.gqa_abi_version.restype = ctypes.c_int32
    assert lib.gqa_abi_version() == 8


def test_debug_library_has_the_nvtx_ranges_and_the_product_library_does_not(debug_lib):
    from sliding_window_gb300 import build
    nm = lambda path: subprocess.run(["nm", path], capture_output=True, text=True).stdout  # noqa: E731
    assert "nvtxRangePushA" in nm(debug_lib) or "nvtxGlobals" in nm(debug_lib)
    product = build.build()
    assert "nvtx" not in nm(product).lower()
    assert "gqa_test_bounds_check" not in nm(product)
