"""Host-side checks of the C ABI. No kernel runs here.

* libmoe.so loads, and it exports every function include/moe.h declares.
* The Guard rejects bad or unsupported configs before touching the device.
* Calls with a NULL plan or bad arguments return status codes and do not crash.
"""
import ctypes
import os
import re

import pytest

import moe_expert_layer_top_gb300 as pkg
from moe_expert_layer_top_gb300 import abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pkg.build.build()
    return abi.load()


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_and_binding_agree(lib):
    assert header_functions() == sorted(abi.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_bounds_checked_library_exports_every_declared_symbol(lib):
    """libmoe_debug.so (the -DMOE_DEBUG_BOUNDS build) has the same ABI."""
    dbg = ctypes.CDLL(pkg.build.DEBUG_LIB_PATH)
    for name in header_functions():
        assert ctypes.cast(getattr(dbg, name), ctypes.c_void_p).value, name
    assert dbg.moe_abi_version() == abi.MOE_ABI_VERSION


def test_abi_version_and_status_strings(lib):
    assert lib.moe_abi_version() == abi.MOE_ABI_VERSION
    assert abi.moe_status_string(abi.MOE_OK) == "MOE_OK"
    assert abi.moe_status_string(abi.MOE_ERR_TIMEOUT) == "MOE_ERR_TIMEOUT"
    assert abi.moe_status_string(99) == "MOE_ERR_UNKNOWN"


def fake_weights(shared=False):
    w = abi.MoeWeights()
    for i, (name, _) in enumerate(abi.MoeWeights._fields_):
        if name.startswith("sh_") and not shared:
            continue
        setattr(w, name, 0x10000 * (i + 1))  # never dereferenced: the Guard fails first or the device part stops
    return w


def cfg(**kw):
    base = dict(hidden=4096, intermediate=2048, num_experts=256, top_k=8, num_shared=0, max_rows=384, flags=0,
                wait_timeout_ns=0, weight_format=0, swiglu_limit=0.0)
    base.update(kw)
    return abi.MoeConfig(**base)


@pytest.mark.parametrize("kw,expect", [
    (dict(hidden=0), abi.MOE_ERR_INVALID_ARG),
    (dict(top_k=0), abi.MOE_ERR_INVALID_ARG),
    (dict(top_k=300), abi.MOE_ERR_INVALID_ARG),          # k > E
    (dict(num_shared=2), abi.MOE_ERR_INVALID_ARG),
    (dict(max_rows=0), abi.MOE_ERR_INVALID_ARG),
    (dict(hidden=32, intermediate=32), abi.MOE_ERR_UNSUPPORTED),
    (dict(hidden=7200), abi.MOE_ERR_UNSUPPORTED),        # not a multiple of 128
    (dict(intermediate=2300), abi.MOE_ERR_UNSUPPORTED),
    (dict(hidden=32768, intermediate=4096), abi.MOE_ERR_UNSUPPORTED),   # above 16384
    (dict(intermediate=2304, flags=abi.MOE_FLAG_PATH_GEMV), abi.MOE_ERR_UNSUPPORTED),  # GEMV: compiled shapes
    (dict(hidden=7168, flags=abi.MOE_FLAG_PATH_GEMV), abi.MOE_ERR_UNSUPPORTED),
    (dict(weight_format=abi.MOE_WEIGHTS_MXFP4, flags=abi.MOE_FLAG_PATH_GEMV), abi.MOE_ERR_UNSUPPORTED),
    (dict(weight_format=2), abi.MOE_ERR_INVALID_ARG),
    (dict(swiglu_limit=float("nan")), abi.MOE_ERR_INVALID_ARG),
    (dict(num_experts=1025, top_k=8), abi.MOE_ERR_UNSUPPORTED),
    (dict(num_experts=64, top_k=33), abi.MOE_ERR_UNSUPPORTED),
    (dict(max_rows=5000), abi.MOE_ERR_UNSUPPORTED),
    (dict(num_experts=1024, max_rows=4096), abi.MOE_ERR_UNSUPPORTED),  # 512 KB of bitmap: beyond shared memory
    (dict(flags=abi.MOE_FLAG_PATH_GEMV | abi.MOE_FLAG_PATH_MMA), abi.MOE_ERR_INVALID_ARG),
])
def test_guard_rejects_before_device(lib, kw, expect):
    st, h = abi.moe_plan_status_code(cfg(**kw), fake_weights())
    assert st == expect and h is None


def test_guard_checks_weight_pointers(lib):
    w = fake_weights()
    w.w_up = None
    assert abi.moe_plan_status_code(cfg(), w)[0] == abi.MOE_ERR_INVALID_ARG
    w = fake_weights()
    w.s_down = 0x10001  # misaligned
    assert abi.moe_plan_status_code(cfg(), w)[0] == abi.MOE_ERR_INVALID_ARG
    # shared pointers must match num_shared
    assert abi.moe_plan_status_code(cfg(num_shared=1), fake_weights(False))[0] == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_plan_status_code(cfg(num_shared=0), fake_weights(True))[0] == abi.MOE_ERR_INVALID_ARG
    # MXFP4 code arrays must be 32-byte aligned (packed 4-bit tensor maps)
    w = fake_weights()
    w.w_gate = 0x10010  # 16-byte but not 32-byte aligned
    assert abi.moe_plan_status_code(cfg(weight_format=abi.MOE_WEIGHTS_MXFP4), w)[0] == abi.MOE_ERR_INVALID_ARG


def test_null_arguments_return_codes(lib):
    assert lib.moe_plan(None, None, None, None) == abi.MOE_ERR_INVALID_ARG
    h = ctypes.c_void_p(123)
    assert lib.moe_plan(ctypes.byref(cfg()), None, None, ctypes.byref(h)) == abi.MOE_ERR_INVALID_ARG
    assert h.value is None  # *plan_out is cleared on failure
    assert lib.moe_forward(None, None, None, 6, None, None, None, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_forward_host(None, None, None, 6, None, None) == abi.MOE_ERR_INVALID_ARG
    io = abi.fused_io()
    assert lib.moe_forward_fused(None, None, 6, ctypes.byref(io), None, None, None, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_destroy(None) == abi.MOE_OK
    assert lib.moe_quantize_mxfp8(None, 4, 48, None, None, None) == abi.MOE_ERR_INVALID_ARG  # cols % 32
    assert lib.moe_quantize_mxfp8(None, 0, 64, None, None, None) == abi.MOE_OK               # empty
    ms, n = ctypes.c_double(), ctypes.c_int32()
    assert lib.moe_kernel_times(None, ctypes.byref(ms), ctypes.byref(n)) == abi.MOE_ERR_INVALID_ARG


def test_binding_refuses_missing_library(tmp_path):
    with pytest.raises(RuntimeError):
        abi.load(str(tmp_path / "libmoe.so"))
