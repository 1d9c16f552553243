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
    # function declarations (a typedef of a function-pointer type is not one)
    return sorted(set(re.findall(r"^\s*(?!typedef\b)(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


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


def _header_enum(name):
    text = open(HEADER).read()
    body = re.search(r"typedef enum " + name + r"\s*\{(.*?)\}", text, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    return {k: int(v) for k, v in re.findall(r"(\w+)\s*=\s*(\d+)", body)}


def test_binding_constants_match_the_header():
    from serving_layer_moe_gb300 import binding as b
    dt = _header_enum("moe_dtype")
    assert dt == {"MOE_F32": 0, "MOE_BF16": 1, "MOE_FP8E4M3_B128": 2, "MOE_NVFP4": 3, "MOE_MXFP4": 4}
    for k, v in dt.items():
        assert getattr(b, k) == v
    assert set(b.DTYPES.values()) == set(dt.values())
    st = _header_enum("moe_status")
    assert {v: k for k, v in st.items()} == b.STATUS


def test_blob_sizes_match_the_header_formula():
    # S as the header states it, against the generator's blob (which the oracle parses)
    from workloads import Shape, make_blob
    H, I = 256, 128
    want = {"f32": 12 * I * H, "bf16": 6 * I * H, "fp8": 3 * I * H + 4 * (2 * I * H + H * I) // 16384,
            "nvfp4": 3 * I * H // 2 + 3 * I * H // 16 + 16, "mxfp4": 3 * I * H // 2 + 3 * I * H // 32}
    for w, S in want.items():
        s = Shape(L=1, E=1, k=1, H=H, I=I, wdtype=w, adtype="bf16")
        assert s.blob_bytes == S and make_blob(s, 1, 0).size == S
        assert S % 16 == (8 if w == "fp8" else 0)     # 6 fp8 scales: 24 bytes


def test_fp4_create_errors_without_a_device_call(lib):
    import ctypes
    from serving_layer_moe_gb300.binding import MOE_MXFP4, MOE_NVFP4, MoEConfigC
    h = ctypes.c_void_p()
    pool = ctypes.create_string_buffer(16)
    for wd in (MOE_NVFP4, MOE_MXFP4):
        # H or I not a multiple of 32
        for hidden, inter in ((264, 128), (256, 136)):
            cfg = MoEConfigC(1, 8, hidden, inter, 2, 4, -1, wd, 1, 0, 1000, 0, 0, 0)
            assert lib.moe_cache_create(ctypes.byref(cfg), pool, 16, None, None, 4, ctypes.byref(h)) == 1
            assert b"fp4" in lib.moe_last_error()


def test_blob_sizes_off_the_16_byte_grid_are_refused_without_a_device_call(lib):
    # fp8 at H=256, I=128 has 6 block scales, so S = 3IH + 24 is 8 bytes off the
    # 16-byte grid every slot and blob must start on
    import ctypes
    from serving_layer_moe_gb300.binding import MOE_FP8E4M3_B128, MoEConfigC
    h = ctypes.c_void_p()
    pool = ctypes.create_string_buffer(16)
    cfg = MoEConfigC(1, 8, 256, 128, 2, 1, -1, MOE_FP8E4M3_B128, 1, 0, 1000, 0, 0, 0)
    assert lib.moe_cache_create(ctypes.byref(cfg), pool, 16, None, None, 4, ctypes.byref(h)) == 1
    assert b"multiple of 16" in lib.moe_last_error()
    assert lib.moe_layer_ffn_noalloc(8, 256, 128, 2, MOE_FP8E4M3_B128, 1, None, 0, None, None, None, None,
                                     None) == 1
    assert b"multiple of 16" in lib.moe_last_error()
    # 512 x 256 has 24 scales: accepted by the shape checks (fails later on the NULL pool)
    cfg = MoEConfigC(1, 8, 512, 256, 2, 1, -1, MOE_FP8E4M3_B128, 1, 0, 1000, 0, 0, 0)
    assert lib.moe_cache_create(ctypes.byref(cfg), None, 0, None, None, 4, ctypes.byref(h)) == 1
    assert b"host_pool" in lib.moe_last_error()


def test_noalloc_refuses_unaligned_pointers_without_a_device_call(lib):
    # the pointers are never dereferenced: the checks run before any CUDA call
    import ctypes
    from serving_layer_moe_gb300.binding import MOE_BF16
    P = ctypes.c_void_p
    good = dict(e=P(0x10000), x=P(0x20000), i=P(0x30000), w=P(0x40000), o=P(0x50000))
    for key, bad, word in (("x", 0x20008, b"16-byte"), ("o", 0x50004, b"16-byte"), ("i", 0x30002, b"4-byte"),
                           ("w", 0x40001, b"4-byte")):
        a = dict(good)
        a[key] = P(bad)
        st = lib.moe_layer_ffn_noalloc(8, 256, 512, 2, MOE_BF16, MOE_BF16, a["e"], 1, a["x"], a["i"], a["w"], a["o"],
                                       None)
        assert st == 1 and word in lib.moe_last_error(), key


def test_binding_refuses_non_contiguous_buffers():
    import numpy as np
    import torch
    from serving_layer_moe_gb300.binding import _ptr
    assert _ptr(None) is None
    a = np.zeros((4, 4), np.float32)
    assert _ptr(a) == a.ctypes.data
    with pytest.raises(ValueError):
        _ptr(a[:, ::2])
    t = torch.zeros(4, 4)
    assert _ptr(t) == t.data_ptr()
    with pytest.raises(ValueError):
        _ptr(t.t())
