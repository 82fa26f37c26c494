"""Number formats of the MoE step: bfloat16, FP8 E4M3 and MXFP8 (group-32 UE8M0).

Oracle module (test infrastructure only). See ``oracle/__init__.py``.

The pages name the formats only. "Beyond Day-0: Optimizing DeepSeek-V4.1
Flash in SGLang", section 2.1, speaks of group-32 FP8 weights and scales in
the Blackwell MXFP8 layout. The definitions here follow the OCP
Microscaling Formats (MX) Specification v1.0:

* E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits. There are no
  infinities. 0x7F and 0xFF are NaN. The largest finite value is 448.
* UE8M0 scale: an 8-bit biased exponent. Its value is 2^(code - 127).
  Code 255 is NaN and is never produced here.
* Shared scale of a 32-element group: 2^(floor(log2(amax)) - emax_elem), with
  emax_elem = 8, the exponent of E4M3's largest normal (448 = 1.75 * 2^8).
  Elements are v / scale, rounded to nearest-even and saturated to +-448.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_EMAX = 8
UE8M0_BIAS = 127
GROUP = 32


# --------------------------------------------------------------------------- bf16

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns: the top half of a binary32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def f32_to_bf16_bits(f) -> np.ndarray:
    """binary32 -> bfloat16, round to nearest, ties to even.

    Overflow rounds to infinity, as IEEE rounding does. NaN maps to a quiet NaN
    with the same sign.
    """
    f = np.asarray(f, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(f)
    if np.any(nan):
        sign = ((u >> np.uint64(16)) & np.uint64(0x8000)).astype(np.uint16)
        r = np.where(nan, sign | np.uint16(0x7FC0), r)
    return r


# --------------------------------------------------------------------------- e4m3

def _e4m3_value(code: int) -> float:
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * m * 2.0 ** -9          # subnormal: (m/8) * 2^(1-7)
    return sign * (8 + m) * 2.0 ** (e - 10)  # normal: (1 + m/8) * 2^(e-7)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)
# Non-negative finite values, codes 0x00..0x7E, strictly increasing from 0 to 448.
_E4M3_POS = E4M3_TABLE[:0x7F].copy()


def e4m3_decode(codes) -> np.ndarray:
    """Value of E4M3 codes (exact in fp64)."""
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(v) -> np.ndarray:
    """Round fp64 values to E4M3: nearest, ties to even mantissa, saturating.

    * |v| > 448 encodes as +-448 (0x7E / 0xFE).
    * The sign is kept for zero results, so -0.0 and negative underflow give 0x80.
    * Inputs must be finite.
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - a
    # The code's lowest bit is the mantissa's lowest bit, so "even" means code % 2 == 0.
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(v), code | np.uint8(0x80), code).astype(np.uint8)


# --------------------------------------------------------------------------- MXFP8

def ue8m0_value(codes) -> np.ndarray:
    """2^(code - 127) for UE8M0 scale codes 0..254."""
    c = np.asarray(codes, dtype=np.int64)
    return np.ldexp(1.0, c - UE8M0_BIAS)


def mxfp8_quantize(v):
    """Quantise along the last axis in groups of 32.

    Returns (q, s). q holds uint8 E4M3 codes, same shape as v. s holds uint8
    UE8M0 codes, with shape [..., n/32].

    For each group:
      amax  = max |v_i|
      code  = 0 if amax == 0, else clamp(floor(log2 amax) - 8 + 127, 0, 254)
      q_i   = e4m3_encode(v_i * 2^(127 - code))    (the scaling is exact)

    floor(log2 amax) is read exactly from frexp: amax = m * 2^ex with m in
    [0.5, 1), so floor(log2 amax) = ex - 1.
    """
    v = np.asarray(v, dtype=np.float64)
    n = v.shape[-1]
    if n % GROUP:
        raise ValueError("last axis must be a multiple of 32")
    g = v.reshape(v.shape[:-1] + (n // GROUP, GROUP))
    amax = np.max(np.abs(g), axis=-1)
    _, ex = np.frexp(amax)
    code = np.clip(ex.astype(np.int64) - 1 - E4M3_EMAX + UE8M0_BIAS, 0, 254)
    code = np.where(amax == 0.0, 0, code)
    scaled = np.ldexp(g, (UE8M0_BIAS - code)[..., None])
    q = e4m3_encode(scaled).reshape(v.shape)
    return q, code.astype(np.uint8)


def mxfp8_dequantize(q, s) -> np.ndarray:
    """Value of MXFP8 data, exact in fp64: e4m3(q_i) * 2^(s_group - 127)."""
    q = np.asarray(q, dtype=np.uint8)
    n = q.shape[-1]
    vals = e4m3_decode(q).reshape(q.shape[:-1] + (n // GROUP, GROUP))
    return (vals * ue8m0_value(s)[..., None]).reshape(q.shape)


# --------------------------------------------------------------------------- e2m1 / MXFP4
# OCP MX v1.0, FP4 element E2M1: 1 sign bit, 2 exponent bits (bias 1), 1
# mantissa bit. There are no infinities or NaNs. The values are
# +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}; the largest is 6 = 1.5 * 2^2, so emax_elem = 2.
# MXFP4 uses the same UE8M0 group-32 scale rule as MXFP8 with emax_elem = 2.
# Two E2M1 codes share a byte: element 2i in the low nibble, 2i+1 in the high
# nibble (the pages name the format, flashinfer_mxfp4 and "MXFP4 weights",
# but not a packing; this is the plainest one and the one sub-byte element
# types commonly use).

E2M1_MAX = 6.0
E2M1_EMAX = 2


def _e2m1_value(code: int) -> float:
    sign = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return sign * m * 0.5                    # subnormal: (m/2) * 2^(1-1)
    return sign * (2 + m) * 2.0 ** (e - 2)       # normal: (1 + m/2) * 2^(e-1)


E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)
_E2M1_POS = E2M1_TABLE[:8].copy()  # codes 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6


def e2m1_decode(codes) -> np.ndarray:
    """Value of E2M1 codes 0..15 (exact in fp64)."""
    return E2M1_TABLE[np.asarray(codes, dtype=np.uint8) & np.uint8(0xF)]


def e2m1_encode(v) -> np.ndarray:
    """Round fp64 values to E2M1 codes 0..15: nearest, ties to even mantissa,
    saturating at +-6, sign of zero kept (negative underflow gives 0x8).
    Inputs must be finite."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), E2M1_MAX)
    hi = np.clip(np.searchsorted(_E2M1_POS, a, side="left"), 0, 7)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _E2M1_POS[lo]
    d_hi = _E2M1_POS[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(v), code | np.uint8(0x8), code).astype(np.uint8)


def pack_e2m1(codes) -> np.ndarray:
    """[..., n] codes (n even) -> [..., n/2] bytes, element 2i in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & np.uint8(0xF)) | ((c[..., 1::2] & np.uint8(0xF)) << np.uint8(4))


def unpack_e2m1(packed) -> np.ndarray:
    """[..., n/2] bytes -> [..., n] codes."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & np.uint8(0xF)
    out[..., 1::2] = p >> np.uint8(4)
    return out


def mxfp4_quantize(v):
    """Quantise along the last axis in groups of 32 to MXFP4.

    Returns (q, s): q holds the packed E2M1 codes, shape [..., n/2] (uint8);
    s the UE8M0 codes, shape [..., n/32].

    For each group:
      amax  = max |v_i|
      code  = 0 if amax == 0, else clamp(floor(log2 amax) - 2 + 127, 0, 254)
      q_i   = e2m1_encode(v_i * 2^(127 - code))    (the scaling is exact)
    """
    v = np.asarray(v, dtype=np.float64)
    n = v.shape[-1]
    if n % GROUP:
        raise ValueError("last axis must be a multiple of 32")
    g = v.reshape(v.shape[:-1] + (n // GROUP, GROUP))
    amax = np.max(np.abs(g), axis=-1)
    _, ex = np.frexp(amax)
    code = np.clip(ex.astype(np.int64) - 1 - E2M1_EMAX + UE8M0_BIAS, 0, 254)
    code = np.where(amax == 0.0, 0, code)
    scaled = np.ldexp(g, (UE8M0_BIAS - code)[..., None])
    q = e2m1_encode(scaled).reshape(v.shape)
    return pack_e2m1(q), code.astype(np.uint8)


def mxfp4_dequantize(q, s) -> np.ndarray:
    """Value of MXFP4 data (packed codes q, scales s), exact in fp64."""
    codes = unpack_e2m1(q)
    n = codes.shape[-1]
    vals = e2m1_decode(codes).reshape(codes.shape[:-1] + (n // GROUP, GROUP))
    return (vals * ue8m0_value(s)[..., None]).reshape(codes.shape)
