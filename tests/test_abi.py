"""The C-ABI library loads and exports every function include/moe_cache.h declares (no GPU needed)."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_cache.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from serving_layer_moe_gb300 import build as b
    if not os.path.exists(b.LIB):
        b.build()
    from serving_layer_moe_gb300 import load_library
    return load_library()


def test_header_declares_the_boundary():
    fns = declared_functions()
    for name in ["moe_cache_create", "moe_cache_resize", "moe_cache_destroy", "moe_layer_decode",
                 "moe_layer_prefill", "bench_bw", "moe_cache_get_state", "moe_last_error"]:
        assert name in fns


def test_library_exports_every_declared_symbol(lib):
    from serving_layer_moe_gb300 import SYMBOLS
    fns = declared_functions()
    assert sorted(SYMBOLS) == fns
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in fns:
        assert name in exported, name
        assert hasattr(lib, name)


def test_errors_without_a_device_call(lib):
    import ctypes
    from serving_layer_moe_gb300.binding import MoEConfigC
    # argument checks happen before any CUDA call
    h = ctypes.c_void_p()
    assert lib.moe_cache_create(None, None, 0, None, None, 1, ctypes.byref(h)) == 1
    assert b"NULL" in lib.moe_last_error()
    cfg = MoEConfigC(1, 8, 256, 512, 2, 4, -1, 0, 0, 0, 0, 0, 0, 0)
    assert lib.moe_cache_create(ctypes.byref(cfg), None, 0, None, None, 4, ctypes.byref(h)) == 1
    assert lib.moe_layer_decode(None, 0, 1, None, None, None, None, None, None, None) == 1
