"""The C-ABI library builds, loads without a GPU and exports every entry point
that include/moe_nvfp4.h declares (no compute calls)."""
import ctypes
import os
import re

import moe_routed_expert_router_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe_nvfp4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(moe.EXPORTS)


def test_library_loads_and_exports_every_symbol():
    L = moe.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert L.moe_version().startswith(b"moe_nvfp4")
    assert L.moe_status_string(4) == b"non-finite activation"


def test_host_side_argument_checks_need_no_gpu():
    L = moe.lib()
    cfg = moe.Config(4096, 1536, 128, 8, 4, 0, 1, 0, 0, 0)
    h = ctypes.c_void_p()
    assert L.moe_plan_create(None, ctypes.byref(h)) == moe.ERR_INVALID_ARG
    bad = moe.Config(4000, 1536, 128, 8, 4, 0, 1, 0, 0, 0)          # H not a multiple of 256
    assert L.moe_plan_create(ctypes.byref(bad), ctypes.byref(h)) == moe.ERR_UNSUPPORTED_SHAPE
    bad = moe.Config(4096, 1536, 4, 8, 4, 0, 1, 0, 0, 0)            # k > E
    assert L.moe_plan_create(ctypes.byref(bad), ctypes.byref(h)) == moe.ERR_UNSUPPORTED_SHAPE
    bad = moe.Config(4096, 1536, 128, 8, 4, 7, 1, 0, 0, 0)          # unknown router kind
    assert L.moe_plan_create(ctypes.byref(bad), ctypes.byref(h)) == moe.ERR_INVALID_ARG
    bad = moe.Config(4096, 1536, 128, 8, 4, 0, 1, 0, 0, 0, 2)       # unknown router word type
    assert L.moe_plan_create(ctypes.byref(bad), ctypes.byref(h)) == moe.ERR_INVALID_ARG
    assert L.moe_convert_f32(None, 16, 7, None, None) == moe.ERR_INVALID_ARG   # unknown format
    assert L.moe_convert_f32(8, 16, moe.FMT_E2M1, 16, None) == moe.ERR_MISALIGNED
    assert L.moe_quantize_nvfp4(None, 1, 4, 24, None, None, None, None) == moe.ERR_UNSUPPORTED_SHAPE
    assert L.moe_quantize_nvfp4(8, 1, 4, 32, 16, 16, 16, None) == moe.ERR_MISALIGNED
    assert L.moe_forward(None, None, 0, None, None, None, None, None, None) == moe.ERR_INVALID_ARG
