"""Seeded synthetic inputs for the small-batch MXFP8 MoE step.

This module only draws numbers. It holds none of the MoE method's arithmetic
(no routing, no quantisation, no GEMM). The oracle and the CUDA path both take
their inputs from here, and nothing else is shared between them.

Counter-based generator
-----------------------
Every value is a pure function of (seed, stream, index). It is the SplitMix64
generator of Steele, Lea and Flood, "Fast splittable pseudorandom number
generators" (OOPSLA 2014), in the form Vigna publishes as ``splitmix64.c``:

* state_i = key + (i + 1) * 0x9E3779B97F4A7C15  (mod 2^64)
* out_i   = mix64(state_i), where mix64 is
  z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31

The per-tensor key is ``mix64(seed * 0x9E3779B97F4A7C15 + stream)``.
Because the generator is counter based, any slice of a tensor can be drawn
on its own, and the CUDA implementation in ``synth/synth.cu`` draws the same
bits on the device. ``tests/test_synth.py`` checks that the two agree bit for bit.

Approximately normal values
---------------------------
A bf16 "normal" value uses only integer sums and one binary32 multiply, so
host and device produce identical bits:

* S = the sum of the four 16-bit fields of out_i, in [0, 262140].
  It has mean 131070 and variance (65536^2 - 1) / 3 (Irwin-Hall, n = 4).
* v = float32(S - 131070) * c, with c = float32(sqrt(3) / 65536 * sigma).
  This is one correctly rounded binary32 multiply.
* The result is v rounded to bfloat16, nearest-even.

The values are bounded by about 3.46 sigma and have unit variance after
scaling. They stand in for "~N(0, sigma)".

Workloads
---------
``WORKLOADS`` lists the five shapes that are measured and parity-tested:
T token rows, hidden H, E routed experts, top-k, intermediate I, an optional
shared expert, and uniform or Zipf(1.1) routing.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK = (1 << 64) - 1

BASE_SEED = 42

# Stream ids of the synthetic tensors.
STREAM_X = 1
STREAM_LOGITS = 2
STREAM_LOGITS_RETRY = 3
# The steps either side of the MoE step: router weight, residual streams,
# RMSNorm weight and per-row stream-mixing coefficients.
STREAM_ROUTER = 4
STREAM_RESID = 5
STREAM_NORM_W = 6
STREAM_MIX_RES = 7
STREAM_MIX_POST = 8
STREAM_MIX_PRE = 9


def stream_gate(e: int) -> int:
    return 1000 + 3 * e


def stream_up(e: int) -> int:
    return 1001 + 3 * e


def stream_down(e: int) -> int:
    return 1002 + 3 * e


# The shared expert's tensors (one shared expert at most).
STREAM_SH_GATE = 900_000
STREAM_SH_UP = 900_001
STREAM_SH_DOWN = 900_002


def mix64_int(z: int) -> int:
    """SplitMix64 finaliser on a Python int (mod 2^64)."""
    z &= _MASK
    z ^= z >> 30
    z = (z * _M1) & _MASK
    z ^= z >> 27
    z = (z * _M2) & _MASK
    z ^= z >> 31
    return z


def stream_key(seed: int, stream: int) -> int:
    """Per-tensor SplitMix64 state offset."""
    return mix64_int((seed * GOLDEN + stream) & _MASK)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(_M1)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(_M2)
    z = z ^ (z >> np.uint64(31))
    return z


def counter_u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """out_i for i in [start, start + count), as uint64."""
    key = np.uint64(stream_key(seed, stream))
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = key + idx * np.uint64(GOLDEN)
        return _mix64(state)


def sigma_constant(sigma: float) -> np.float32:
    """c = float32(sqrt(3) / 65536 * sigma), the single multiplier of the draw."""
    return np.float32(math.sqrt(3.0) / 65536.0 * sigma)


def _f32_to_bf16_rne(v: np.ndarray) -> np.ndarray:
    u = v.astype(np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    return ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def normal_bf16(seed: int, stream: int, start: int, count: int, sigma: float) -> np.ndarray:
    """Approximately N(0, sigma) values as bf16 bit patterns (uint16)."""
    h = counter_u64(seed, stream, start, count)
    m16 = np.uint64(0xFFFF)
    s = (h & m16) + ((h >> np.uint64(16)) & m16) + ((h >> np.uint64(32)) & m16) + (h >> np.uint64(48))
    centred = (s.astype(np.int64) - 131070).astype(np.float32)  # exact: |.| <= 131070 < 2^24
    v = centred * sigma_constant(sigma)  # one binary32 multiply
    return _f32_to_bf16_rne(v)


def uniform_open01(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Uniform doubles in (0, 1): (top 53 bits + 0.5) * 2^-53."""
    h = counter_u64(seed, stream, start, count)
    return ((h >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    shared: int  # 0 or 1
    routing: str  # "uniform" or "zipf"
    zipf_s: float = 1.1
    description: str = ""
    fmt: str = "mxfp8"          # expert weight format: "mxfp8" or "mxfp4"
    swiglu_limit: float = 0.0   # clipped SwiGLU limit (<= 0: no clip)

    @property
    def expert_bytes(self) -> int:
        """Weight bytes of one expert: 3 matrices of I x H codes (1 byte each for
        MXFP8, half a byte for MXFP4) plus one scale byte per 32."""
        if self.fmt == "mxfp4":
            return 3 * self.I * self.H * 17 // 32
        return 3 * self.I * self.H * 33 // 32


WORKLOADS = {
    "tiny": Workload("tiny", 6, 512, 8, 2, 256, 0, "uniform",
                     description="tiny MoE step: T=6, H=512, E=8, top-2, I=256"),
    "bs1": Workload("bs1", 6, 4096, 256, 8, 2048, 0, "uniform",
                    description="bs1 speculative-verify shape: T=6, H=4096, E=256, top-8, I=2048"),
    "bs4": Workload("bs4", 24, 4096, 256, 8, 2048, 0, "uniform",
                    description="bs4 verify shape: T=24, H=4096, E=256, top-8, I=2048"),
    "bs16": Workload("bs16", 96, 4096, 256, 8, 2048, 0, "zipf",
                     description="bs16 verify shape: T=96, Zipf(1.1) routing"),
    "bs64": Workload("bs64", 384, 4096, 256, 8, 2048, 1, "zipf",
                     description="bs64 verify shape: T=384, E=256 + 1 shared expert, Zipf(1.1) routing"),
    # the pages' checkpoint format: MXFP4 expert weights, I = 4 x 576, clipped SwiGLU (limit not given; 7.0 here)
    "bs1_fp4": Workload("bs1_fp4", 6, 4096, 256, 8, 2304, 0, "uniform", fmt="mxfp4", swiglu_limit=7.0,
                        description="bs1 shape with MXFP4 weights, I=2304, clipped SwiGLU"),
    "bs4_fp4": Workload("bs4_fp4", 24, 4096, 256, 8, 2304, 0, "uniform", fmt="mxfp4", swiglu_limit=7.0,
                        description="bs4 shape with MXFP4 weights, I=2304, clipped SwiGLU"),
    "bs64_fp4": Workload("bs64_fp4", 384, 4096, 256, 8, 2304, 1, "zipf", fmt="mxfp4", swiglu_limit=7.0,
                         description="bs64 shape with MXFP4 weights, I=2304, clipped SwiGLU"),
}


def x_bf16(seed: int, T: int, H: int) -> np.ndarray:
    """Token rows x ~ N(0, 1) as bf16 bits, [T][H]."""
    return normal_bf16(seed, STREAM_X, 0, T * H, 1.0).reshape(T, H)


def _row_margin_ok(row: np.ndarray, k: int, margin: float) -> bool:
    s = np.sort(row.astype(np.float64))[::-1]
    gaps = s[: k] - s[1: k + 1]
    return bool(np.all(gaps >= margin))


def router_logits(seed: int, T: int, E: int, k: int, routing: str = "uniform",
                  zipf_s: float = 1.1, margin: float = 1e-3) -> np.ndarray:
    """Router logits fp32 [T][E]: log p_e + Gumbel(0, 1).

    The top-k of log p + Gumbel noise samples k experts without replacement
    with probability proportional to p (Kool, van Hoof and Welling, ICML 2019).
    Uniform routing uses p_e = 1/E. Zipf routing uses p_e proportional to
    (e + 1)^-s, so expert 0 is the most popular.
    A row whose sorted gaps among the first k + 1 values fall below ``margin``
    is drawn again from a retry stream, until every such gap is at least
    ``margin``. The drawn values are exact IEEE doubles rounded once to fp32.
    """
    if routing == "uniform":
        logp = np.full(E, -math.log(E))
    elif routing == "zipf":
        w = (np.arange(E, dtype=np.float64) + 1.0) ** (-zipf_s)
        logp = np.log(w / w.sum())
    else:
        raise ValueError(f"unknown routing {routing!r}")
    out = np.empty((T, E), dtype=np.float32)
    u = uniform_open01(seed, STREAM_LOGITS, 0, T * E).reshape(T, E)
    for t in range(T):
        row = (logp - np.log(-np.log(u[t]))).astype(np.float32)
        attempt = 0
        while not _row_margin_ok(row, min(k, E - 1), margin):
            attempt += 1
            if attempt > 1000:
                raise RuntimeError("could not draw a row with the requested margin")
            ur = uniform_open01(seed, STREAM_LOGITS_RETRY, (attempt * (1 << 20) + t) * E, E)
            row = (logp - np.log(-np.log(ur))).astype(np.float32)
        out[t] = row
    return out


def expert_sigma(fan_in: int) -> float:
    """Weights ~ N(0, 1/sqrt(fan_in))."""
    return 1.0 / math.sqrt(fan_in)


def expert_weight_bf16(seed: int, stream: int, rows: int, cols: int,
                       row_start: int = 0, row_count: int | None = None) -> np.ndarray:
    """Rows [row_start, row_start + row_count) of a [rows][cols] weight matrix,
    drawn ~ N(0, 1/sqrt(cols)) as bf16 bits. cols is the fan-in (the K axis)."""
    if row_count is None:
        row_count = rows - row_start
    flat = normal_bf16(seed, stream, row_start * cols, row_count * cols, expert_sigma(cols))
    return flat.reshape(row_count, cols)


def bf16_bits_to_float32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (a format conversion, no rounding)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def router_weight_bf16(seed: int, E: int, H: int) -> np.ndarray:
    """Router weight W_r ~ N(0, 1/sqrt(H)) as bf16 bits, [E][H]. With x ~ N(0, 1)
    the projected logits have about unit variance."""
    return normal_bf16(seed, STREAM_ROUTER, 0, E * H, expert_sigma(H)).reshape(E, H)


def residual_bf16(seed: int, T: int, S: int, H: int) -> np.ndarray:
    """S residual streams per token row, ~ N(0, 1) as bf16 bits, [T][S][H]."""
    return normal_bf16(seed, STREAM_RESID, 0, T * S * H, 1.0).reshape(T, S, H)


def norm_weight_bf16(seed: int, H: int) -> np.ndarray:
    """RMSNorm weight gamma ~ 1 + N(0, 0.25) as bf16 bits, [H]: the normal draw,
    plus 1.0 in binary32, rounded to bf16 (nearest even)."""
    d = bf16_bits_to_float32(normal_bf16(seed, STREAM_NORM_W, 0, H, 0.25))
    return _f32_to_bf16_rne(d + np.float32(1.0))


def mix_coefficients(seed: int, T: int, S: int):
    """Per-row stream-mixing coefficients, fp32:
    res [T][S][S] uniform in (0, 2/S) (each row of the matrix sums to about 1),
    post [T][S] uniform in (0, 2), pre [T][S] uniform in (0, 1)."""
    res = (uniform_open01(seed, STREAM_MIX_RES, 0, T * S * S) * (2.0 / S)).astype(np.float32)
    post = (uniform_open01(seed, STREAM_MIX_POST, 0, T * S) * 2.0).astype(np.float32)
    pre = uniform_open01(seed, STREAM_MIX_PRE, 0, T * S).astype(np.float32)
    return res.reshape(T, S, S), post.reshape(T, S), pre.reshape(T, S)


# ----------------------------------------------------------------- structured inputs for exact parity

STREAM_EXACT = 11
STREAM_OUTLIER = 12


def _f32_to_bf16_exact(v: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of float32 values that bf16 represents exactly."""
    u = np.asarray(v, dtype=np.float32).view(np.uint32)
    if np.any(u & np.uint32(0xFFFF)):
        raise ValueError("value not representable in bf16")
    return (u >> np.uint32(16)).astype(np.uint16)


def _grid(seed: int, stream: int, rows: int, cols: int, base_choices, signed: bool) -> np.ndarray:
    """[rows][cols] float32 values m * 2^(a - d): per row and 32-column group a
    base exponent a from base_choices, per element m in {1, 1.5} and d in
    {0, 1, 2} (and a sign when signed). A group then spans a factor of 6 at
    most: every value is exact in bf16, in E4M3 and in E2M1 at the group's
    shared power-of-two scale."""
    groups = cols // 32
    hb = counter_u64(seed, stream, 0, rows * groups).reshape(rows, groups)
    base = np.asarray(base_choices, dtype=np.int64)[(hb % np.uint64(len(base_choices))).astype(np.int64)]
    he = counter_u64(seed, stream + 1, 0, rows * cols).reshape(rows, cols)
    m = np.where((he & np.uint64(1)) != 0, 1.5, 1.0)
    d = ((he >> np.uint64(1)) % np.uint64(3)).astype(np.int64)
    s = np.where(signed & ((he >> np.uint64(8)) & np.uint64(1) != 0), -1.0, 1.0)
    a = np.repeat(base, 32, axis=1)
    return (s * m * np.exp2(a - d)).astype(np.float32)


def exact_case(seed: int, T: int, H: int, E: int, k: int, I: int, shared: int = 0, routing: str = "uniform"):
    """Inputs on which every intermediate of the MoE step is exactly defined.

    Token rows and weights take grid values (_grid), so every product of two
    of them is a multiple of 2^-8, and every sum of H (or I) of them stays
    below 2^24 of that unit: the binary32 sums are exact in any order. Per
    expert:
      gate row i = 2^(L_j + b_i) * r_g, with one positive row pattern r_g,
                   b_i in {0, 1} and a level L_j in {0, 1, 2} per 32-row group j;
      up row i   = +-r_u, with one signed row pattern r_u;
      down       = independent signed grid values.
    The token rows are positive, so each gate sum is at least H / 64, far into
    the range where silu(g) rounds to g in binary32. A row's h values are then
    +-2^(L_j + b_i) times one value: h's MXFP8 scale codes differ from group to
    group along I, its groups are exact multiples of a common unit, and the
    down sums are exact too.
    Returns x (bf16 bits [T][H]), logits (fp32 [T][E]) and the bf16 bits of
    gate [E][I][H], up [E][I][H], down [E][H][I] (+ sh_gate, sh_up, sh_down
    when shared)."""
    x = _grid(seed, STREAM_EXACT * 1000, T, H, (-1, 0, 1), False)

    def expert(base_stream):
        rg = _grid(seed, base_stream, 1, H, (-1, 0, 1), False)
        ru = _grid(seed, base_stream + 2, 1, H, (-1, 0, 1), True)
        hb = counter_u64(seed, base_stream + 4, 0, I + I // 32)
        b = (hb[:I] & np.uint64(1)).astype(np.float32)
        level = np.repeat((hb[I:] % np.uint64(3)).astype(np.float32), 32)
        sgn = np.where(((hb[:I] >> np.uint64(1)) & np.uint64(1)) != 0, -1.0, 1.0).astype(np.float32)
        gate = np.exp2(level + b)[:, None] * rg
        up = sgn[:, None] * ru
        down = _grid(seed, base_stream + 5, H, I, (-1, 0), True)
        return _f32_to_bf16_exact(gate), _f32_to_bf16_exact(up), _f32_to_bf16_exact(down)

    parts = [expert(STREAM_EXACT * 1000 + 10 * (e + 1)) for e in range(E)]
    out = {
        "x": _f32_to_bf16_exact(x),
        "logits": router_logits(seed, T, E, k, routing),
        "gate": np.stack([p[0] for p in parts]),
        "up": np.stack([p[1] for p in parts]),
        "down": np.stack([p[2] for p in parts]),
    }
    if shared:
        out["sh_gate"], out["sh_up"], out["sh_down"] = expert(STREAM_EXACT * 1000 + 10 * (E + 1))
    return out


def x_bf16_outliers(seed: int, T: int, H: int, every: int = 97, lo: int = 4, hi: int = 12) -> np.ndarray:
    """Token rows x ~ N(0, 1) (x_bf16) with about one element in `every`
    multiplied by 2^s, s drawn from [lo, hi]: activation outliers that spread
    the exponents inside a 32-group. A power-of-two factor is exact in bf16."""
    x = bf16_bits_to_float32(x_bf16(seed, T, H)).reshape(-1)
    h = counter_u64(seed, STREAM_OUTLIER, 0, T * H)
    pick = (h % np.uint64(every)) == 0
    s = (lo + ((h >> np.uint64(16)) % np.uint64(hi - lo + 1)).astype(np.int64)).astype(np.float32)
    x = np.where(pick, x * np.exp2(s), x).astype(np.float32)
    return _f32_to_bf16_exact(x).reshape(T, H)
