"""Device side of the seeded generator: loads synth/_build/libmoe_synth.so.

It draws the same bits as ``synth.normal_bf16`` into device memory, for the
large weight tensors that are too slow to draw on the host. Numbers only; no
method arithmetic.
"""
from __future__ import annotations

import ctypes
import os

import synth

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libmoe_synth.so")
_lib = None


def load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"generator library not built: {LIB_PATH}")
        lib = ctypes.CDLL(LIB_PATH)
        lib.synth_normal_bf16.restype = ctypes.c_int
        lib.synth_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float,
                                          ctypes.c_void_p, ctypes.c_void_p]
        _lib = lib
    return _lib


def normal_bf16(seed: int, stream_id: int, start: int, count: int, sigma: float, out_ptr: int, cuda_stream=None):
    """Device twin of synth.normal_bf16: writes count bf16 values to out_ptr."""
    key = synth.stream_key(seed, stream_id)
    c = float(synth.sigma_constant(sigma))
    rc = load().synth_normal_bf16(key, start, count, c, out_ptr, cuda_stream)
    if rc != 0:
        raise RuntimeError(f"synth_normal_bf16 launch failed: cudaError {rc}")
