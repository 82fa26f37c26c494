"""Thin ctypes binding of the C ABI in include/moe.h (argument marshalling only).

Every step of the MoE computation runs in the CUDA kernels of libmoe.so. This
module only loads the library, mirrors its structs, and converts pointers
(ints, or torch tensors through ``data_ptr()``) and status codes. If the
library is missing, loading fails loudly; there is no other code path.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

MOE_ABI_VERSION = 3

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_OOM = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE_BOUNDS = 6

MOE_WEIGHTS_MXFP8 = 0
MOE_WEIGHTS_MXFP4 = 1

MOE_FLAG_TIMING = 1 << 0
MOE_FLAG_PATH_GEMV = 1 << 1
MOE_FLAG_PATH_MMA = 1 << 2
MOE_FLAG_TEST_SKIP_READY = 1 << 8
MOE_FLAG_TEST_BOUNDS = 1 << 9

# Every function declared in include/moe.h.
EXPORTED = (
    "moe_abi_version",
    "moe_status_string",
    "moe_plan",
    "moe_forward",
    "moe_forward_dev",
    "moe_forward_fused",
    "moe_forward_host",
    "moe_quantize_mxfp8",
    "moe_quantize_mxfp4",
    "moe_kernel_times",
    "moe_plan_status",
    "moe_plan_diagnostics",
    "moe_forward_static_scratch",
    "moe_destroy",
)

MOE_STATIC_SCRATCH_BYTES = 8 << 20


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int, lib=None):
        name = lib.moe_status_string(status).decode() if lib is not None else str(status)
        super().__init__(f"{fn} returned {name} ({status})")
        self.status = status


class MoeConfig(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int32),
        ("intermediate", ctypes.c_int32),
        ("num_experts", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("num_shared", ctypes.c_int32),
        ("max_rows", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
        ("wait_timeout_ns", ctypes.c_int64),
        ("weight_format", ctypes.c_uint32),
        ("swiglu_limit", ctypes.c_float),
    ]


_P = ctypes.c_void_p


class MoeWeights(ctypes.Structure):
    _fields_ = [(n, _P) for n in ("w_gate", "s_gate", "w_up", "s_up", "w_down", "s_down",
                                  "sh_w_gate", "sh_s_gate", "sh_w_up", "sh_s_up", "sh_w_down", "sh_s_down")]


class MoeTaps(ctypes.Structure):
    _fields_ = [(n, _P) for n in ("topk_ids", "topk_w", "bitmap", "counts", "slot", "xq", "xs",
                                  "h_bf16", "hq", "hs", "o")]


class MoeFusedIO(ctypes.Structure):
    _fields_ = [
        ("w_router", _P),
        ("logits", _P),
        ("num_streams", ctypes.c_int32),
        ("resid_in", _P),
        ("resid_out", _P),
        ("mix_res", _P),
        ("mix_post", _P),
        ("mix_pre", _P),
        ("norm_weight", _P),
        ("rms_eps", ctypes.c_float),
        ("zq", _P),
        ("zs", _P),
        ("z", _P),
    ]


_lib = None


def library_path() -> str:
    """libmoe.so, or the bounds-checked libmoe_debug.so when MOE_DEBUG_BOUNDS=1."""
    return _build.DEBUG_LIB_PATH if os.environ.get("MOE_DEBUG_BOUNDS") == "1" else _build.LIB_PATH


def load(path: str | None = None):
    """Load libmoe.so (built in-tree by ``build()``) and declare its signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or library_path()
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} (run __graft_entry__.build())")
    lib = ctypes.CDLL(p)
    lib.moe_abi_version.restype = ctypes.c_int32
    lib.moe_abi_version.argtypes = []
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_status_string.argtypes = [ctypes.c_int]
    lib.moe_plan.restype = ctypes.c_int
    lib.moe_plan.argtypes = [ctypes.POINTER(MoeConfig), ctypes.POINTER(MoeWeights), _P, ctypes.POINTER(_P)]
    lib.moe_forward.restype = ctypes.c_int
    lib.moe_forward.argtypes = [_P, _P, _P, ctypes.c_int32, _P, ctypes.POINTER(MoeTaps), _P, _P]
    lib.moe_forward_host.restype = ctypes.c_int
    lib.moe_forward_host.argtypes = [_P, _P, _P, ctypes.c_int32, _P, _P]
    lib.moe_quantize_mxfp8.restype = ctypes.c_int
    lib.moe_quantize_mxfp8.argtypes = [_P, ctypes.c_int64, ctypes.c_int32, _P, _P, _P]
    lib.moe_quantize_mxfp4.restype = ctypes.c_int
    lib.moe_quantize_mxfp4.argtypes = [_P, ctypes.c_int64, ctypes.c_int32, _P, _P, _P]
    lib.moe_kernel_times.restype = ctypes.c_int
    lib.moe_kernel_times.argtypes = [_P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int32)]
    lib.moe_plan_status.restype = ctypes.c_int
    lib.moe_plan_status.argtypes = [_P, ctypes.POINTER(ctypes.c_int32)]
    lib.moe_plan_diagnostics.restype = ctypes.c_int
    lib.moe_plan_diagnostics.argtypes = [_P, ctypes.POINTER(ctypes.c_int64)]
    lib.moe_forward_dev.restype = ctypes.c_int
    lib.moe_forward_dev.argtypes = [_P, _P, _P, _P, _P, _P, _P]
    lib.moe_forward_fused.restype = ctypes.c_int
    lib.moe_forward_fused.argtypes = [_P, _P, ctypes.c_int32, ctypes.POINTER(MoeFusedIO), _P,
                                      ctypes.POINTER(MoeTaps), _P, _P]
    lib.moe_forward_static_scratch.restype = ctypes.c_int
    lib.moe_forward_static_scratch.argtypes = [ctypes.POINTER(MoeConfig), ctypes.POINTER(MoeWeights), _P, _P,
                                               ctypes.c_int32, _P, _P, _P]
    lib.moe_destroy.restype = ctypes.c_int
    lib.moe_destroy.argtypes = [_P]
    if lib.moe_abi_version() != MOE_ABI_VERSION:
        raise RuntimeError("libmoe.so ABI version mismatch")
    if path is None:
        _lib = lib
    return lib


def ptr(x) -> int | None:
    """Raw address of a torch tensor (data_ptr), an int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def stream_ptr(stream) -> int | None:
    """cudaStream_t of a torch.cuda.Stream (or an int handle, or None for the legacy default stream)."""
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def check(fn: str, status: int):
    if status != MOE_OK:
        raise MoeError(fn, status, _lib)


# ----------------------------------------------------------------------------- entry points

def moe_abi_version() -> int:
    return load().moe_abi_version()


def moe_status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


def moe_plan(config: MoeConfig, weights: MoeWeights, stream=None) -> int:
    """Guard + Build. Returns the plan handle; raises MoeError on a non-OK status."""
    lib = load()
    h = _P()
    check("moe_plan", lib.moe_plan(ctypes.byref(config), ctypes.byref(weights), stream_ptr(stream), ctypes.byref(h)))
    return h.value


def moe_plan_status_code(config: MoeConfig, weights: MoeWeights, stream=None) -> tuple[int, int | None]:
    """moe_plan returning (status, handle or None) instead of raising."""
    lib = load()
    h = _P()
    s = lib.moe_plan(ctypes.byref(config), ctypes.byref(weights), stream_ptr(stream), ctypes.byref(h))
    return s, h.value


def moe_forward(plan: int, x, logits, T: int, y, taps: MoeTaps | None = None, d_status=None, stream=None) -> int:
    """Runtime: enqueue one MoE step. Returns the host-side status (raises nothing)."""
    lib = load()
    return lib.moe_forward(plan, ptr(x), ptr(logits), T, ptr(y), ctypes.byref(taps) if taps is not None else None,
                           ptr(d_status), stream_ptr(stream))


def moe_forward_host(plan: int, x_host, logits_host, T: int, y_host, stream=None) -> int:
    """One step from host buffers (synchronous). Returns the step's status."""
    lib = load()
    return lib.moe_forward_host(plan, ptr(x_host), ptr(logits_host), T, ptr(y_host), stream_ptr(stream))


def moe_quantize_mxfp8(x, rows: int, cols: int, q, s, stream=None) -> int:
    return load().moe_quantize_mxfp8(ptr(x), rows, cols, ptr(q), ptr(s), stream_ptr(stream))


def moe_quantize_mxfp4(x, rows: int, cols: int, q, s, stream=None) -> int:
    return load().moe_quantize_mxfp4(ptr(x), rows, cols, ptr(q), ptr(s), stream_ptr(stream))


def moe_kernel_times(plan: int) -> tuple[float, int]:
    lib = load()
    ms = ctypes.c_double()
    n = ctypes.c_int32()
    check("moe_kernel_times", lib.moe_kernel_times(plan, ctypes.byref(ms), ctypes.byref(n)))
    return ms.value, n.value


def moe_plan_status(plan: int) -> int:
    lib = load()
    v = ctypes.c_int32()
    check("moe_plan_status", lib.moe_plan_status(plan, ctypes.byref(v)))
    return v.value


def moe_plan_diagnostics(plan: int) -> list[int]:
    lib = load()
    out = (ctypes.c_int64 * 8)()
    check("moe_plan_diagnostics", lib.moe_plan_diagnostics(plan, out))
    return list(out)


def moe_forward_dev(plan, x, logits, d_T, y, d_status=None, stream=None) -> int:
    """One MoE step whose row count is read from device memory (int32 at d_T)."""
    lib = load()
    return lib.moe_forward_dev(plan, ptr(x), ptr(logits), ptr(d_T), ptr(y), ptr(d_status), stream_ptr(stream))


def fused_io(w_router=None, logits=None, num_streams: int = 0, resid_in=None, resid_out=None, mix_res=None,
             mix_post=None, mix_pre=None, norm_weight=None, rms_eps: float = 0.0, zq=None, zs=None,
             z=None) -> MoeFusedIO:
    """A moe_fused_io_t from tensors (or addresses, or None)."""
    return MoeFusedIO(ptr(w_router), ptr(logits), num_streams, ptr(resid_in), ptr(resid_out), ptr(mix_res),
                      ptr(mix_post), ptr(mix_pre), ptr(norm_weight), rms_eps, ptr(zq), ptr(zs), ptr(z))


def moe_forward_fused(plan, x, T: int, io: MoeFusedIO, y, taps: MoeTaps | None = None, d_status=None,
                      stream=None) -> int:
    """One MoE step with the fused router projection and residual-stream epilogue."""
    lib = load()
    return lib.moe_forward_fused(plan, ptr(x), T, ctypes.byref(io) if io is not None else None, ptr(y),
                                 ctypes.byref(taps) if taps is not None else None, ptr(d_status),
                                 stream_ptr(stream))


def moe_forward_static_scratch(config: MoeConfig, weights: MoeWeights, x, logits, T: int, y, d_status=None,
                               stream=None) -> int:
    """One MoE step with no allocation (scratch in the library's fixed device array)."""
    lib = load()
    return lib.moe_forward_static_scratch(ctypes.byref(config), ctypes.byref(weights), ptr(x), ptr(logits), T, ptr(y),
                                          ptr(d_status), stream_ptr(stream))


def moe_destroy(plan: int | None) -> int:
    return load().moe_destroy(plan)
