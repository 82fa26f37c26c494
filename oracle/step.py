"""The whole MoE step: route, place, quantise x, expert SwiGLU MLPs, combine.

Oracle module (test infrastructure only). See ``oracle/__init__.py``.

Passages followed:

* "FlyDSL Mono Kernels for High-Interactivity LLM Serving in ATOM", section
  "MiniMax-M3: Connecting Attention and Experts". Each expert does an
  up/gate projection and a down projection.
* "Beyond Day-0: Optimizing DeepSeek-V4.1 Flash in SGLang":
  - section 2.1: MXFP8 activation quantisation, and the weighted reduction of
    expert outputs fused with the shared-expert addition;
  - section 3.1: the SwiGLU keeps the original intermediate rounding.

Readings where the pages are silent:

* Intermediate rounding. g and u are rounded to bf16, as an unfused GEMM
  would store them. silu(g)*u is formed in fp64 and rounded to fp32, then to
  bf16. That h is quantised to MXFP8 along I before the down projection.
* SwiGLU clip ("clipped SwiGLU", same page, section 3.1; the limit is not
  given): with a limit L > 0 the bf16-rounded gate is clamped from above,
  g' = min(g, L), and the up projection on both sides, u' = clamp(u, -L, L),
  before h = silu(g') * u'. L <= 0 means no clip (the default).
* Weight format: MXFP8 (E4M3 + UE8M0 per 32) by default; MXFP4 (E2M1 +
  UE8M0 per 32, two codes per byte) for the pages' flashinfer_mxfp4 runner
  ("SGLang's Low-Latency Mode ..." launch command) and "Beyond Day-0" 3.1's
  MXFP4 expert weights. Activations stay MXFP8 either way.
* GEMMs: every product of two MXFP8 values is exact in fp64. The sum over K
  is an fp64 matrix product (a library primitive). The result is rounded to
  fp32, the type the device accumulates in.
* Combine: y[t] = bf16( ((w_1*o_1 + w_2*o_2) + ...) + o_shared ), in binary32,
  in rank order. The shared expert takes every row with weight 1.0.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Mapping

import numpy as np

from .formats import (bf16_bits_to_f64, f32_to_bf16_bits, mxfp4_dequantize, mxfp4_quantize,
                      mxfp8_dequantize, mxfp8_quantize)
from .routing import placement, softmax_topk_weights, topk_ids


@dataclass
class ExpertWeights:
    """One expert's weights in the canonical K-contiguous layout.

    fmt "mxfp8":
      w_gate, w_up: uint8 E4M3 [I][H]; s_gate, s_up: uint8 UE8M0 [I][H/32]
      w_down:       uint8 E4M3 [H][I]; s_down:       uint8 UE8M0 [H][I/32]
    fmt "mxfp4": the same, with w_* holding packed E2M1 codes [rows][K/2].
    """
    w_gate: np.ndarray
    s_gate: np.ndarray
    w_up: np.ndarray
    s_up: np.ndarray
    w_down: np.ndarray
    s_down: np.ndarray
    fmt: str = "mxfp8"

    def dequant(self, which: str) -> np.ndarray:
        """Exact fp64 value of one weight matrix ("gate", "up" or "down")."""
        q, s = getattr(self, "w_" + which), getattr(self, "s_" + which)
        return mxfp4_dequantize(q, s) if self.fmt == "mxfp4" else mxfp8_dequantize(q, s)


def expert_weights_from_bf16(g_bits, u_bits, d_bits, fmt: str = "mxfp8") -> ExpertWeights:
    """Quantise one expert's bf16 weights (bit patterns: gate [I][H], up [I][H],
    down [H][I]) with the oracle's own MXFP8 (or MXFP4) rule along K."""
    quant = mxfp4_quantize if fmt == "mxfp4" else mxfp8_quantize
    wg, sgc = quant(bf16_bits_to_f64(np.asarray(g_bits, dtype=np.uint16)))
    wu, suc = quant(bf16_bits_to_f64(np.asarray(u_bits, dtype=np.uint16)))
    wd, sdc = quant(bf16_bits_to_f64(np.asarray(d_bits, dtype=np.uint16)))
    return ExpertWeights(wg, sgc, wu, suc, wd, sdc, fmt)


def expert_weights_from_synth(seed: int, e, H: int, I: int, fmt: str = "mxfp8") -> ExpertWeights:
    """Draw expert e's bf16 weights from the seeded generator, then quantise
    them with the oracle's own MXFP8 (or MXFP4) rule. e == "shared" selects
    the shared expert."""
    import synth
    if e == "shared":
        sg, su, sd = synth.STREAM_SH_GATE, synth.STREAM_SH_UP, synth.STREAM_SH_DOWN
    else:
        sg, su, sd = synth.stream_gate(e), synth.stream_up(e), synth.stream_down(e)
    return expert_weights_from_bf16(synth.expert_weight_bf16(seed, sg, I, H),
                                    synth.expert_weight_bf16(seed, su, I, H),
                                    synth.expert_weight_bf16(seed, sd, H, I), fmt)


def _round_f32(v) -> np.ndarray:
    return np.asarray(v, dtype=np.float64).astype(np.float32)


def expert_mlp(xq, xs, w: ExpertWeights, swiglu_limit: float = 0.0):
    """SwiGLU expert MLP on MXFP8 token rows xq/xs [n][H].

    swiglu_limit > 0 clips the bf16 gate to <= L and the bf16 up projection
    to [-L, L] before the activation (L taken as a binary32 value).

    Returns g_bf16, u_bf16, h_bf16 ([n][I] bf16 bits; g and u before the
    clip), the MXFP8 quantised h (hq [n][I], hs [n][I/32]) and o (fp32 [n][H]).
    """
    x = mxfp8_dequantize(xq, xs)                              # exact, fp64 [n][H]
    wg = w.dequant("gate")                                    # [I][H]
    wu = w.dequant("up")
    g = f32_to_bf16_bits(_round_f32(x @ wg.T))                # gate projection
    u = f32_to_bf16_bits(_round_f32(x @ wu.T))                # up projection
    gf = bf16_bits_to_f64(g)
    uf = bf16_bits_to_f64(u)
    if swiglu_limit > 0:
        lim = float(np.float32(swiglu_limit))
        gf = np.minimum(gf, lim)                              # clipped SwiGLU
        uf = np.clip(uf, -lim, lim)
    silu = gf / (1.0 + np.exp(-gf))                           # SiLU(g) = g * sigmoid(g)
    h = f32_to_bf16_bits(_round_f32(silu * uf))               # SwiGLU: SiLU(gate) * up
    hq, hs = mxfp8_quantize(bf16_bits_to_f64(h))
    wd = w.dequant("down")                                    # [H][I]
    o = _round_f32(mxfp8_dequantize(hq, hs) @ wd.T)           # down projection
    return g, u, h, hq, hs, o


def moe_route(x_bits, logits, k: int):
    """The step's front: top-k ids, combine weights, placement and the MXFP8
    token rows. Returns a dict with ids, w, bitmap, counts, tiles,
    slot_e/slot_tile/slot_row, rows_of, xq and xs."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    logits = np.asarray(logits, dtype=np.float32)
    E = logits.shape[1]
    ids = topk_ids(logits, k)
    w = softmax_topk_weights(logits, ids)
    plc = placement(ids, E)
    xq, xs = mxfp8_quantize(bf16_bits_to_f64(x_bits))
    return {"ids": ids, "w": w, "xq": xq, "xs": xs, **plc}


def pair_token(p: int, T: int, k: int) -> int:
    """Token row of pair p (routed pairs t*k + j, then shared pairs T*k + t)."""
    return p // k if p < T * k else p - T * k


def expert_pairs(route: dict, T: int, k: int, e, rows=None):
    """Pair ids that expert e (or "shared") serves, restricted to the token
    rows in `rows` (None: all), in rank order."""
    row_set = None if rows is None else set(int(r) for r in rows)
    if e == "shared":
        src = range(T * k, T * k + T)
    else:
        src = (int(p) for p in route["rows_of"][e])
    return [p for p in src if row_set is None or pair_token(p, T, k) in row_set]


def combine(w, o_all, T: int, k: int, shared: bool, rows=None):
    """y[t] = bf16( ((w_1*o_1 + w_2*o_2) + ...) + o_shared ) in binary32, rank
    order; o_all is indexed by pair id. Rows outside `rows` are 0."""
    H = o_all.shape[1]
    y = np.zeros((T, H), dtype=np.uint16)
    for t in (range(T) if rows is None else sorted(set(int(r) for r in rows))):
        acc = w[t, 0] * o_all[t * k + 0]                          # binary32 products and sums
        for j in range(1, k):
            acc = acc + w[t, j] * o_all[t * k + j]
        if shared:
            acc = acc + o_all[T * k + t]
        y[t] = f32_to_bf16_bits(acc.astype(np.float32))
    return y


def moe_step(x_bits, logits, k: int,
             experts: Mapping[int, ExpertWeights] | Callable[[int], ExpertWeights],
             shared: ExpertWeights | None = None,
             rows=None, swiglu_limit: float = 0.0):
    """One MoE step over T token rows.

    x_bits: bf16 bit patterns uint16 [T][H]; logits: fp32 [T][E].
    experts: a mapping or callable giving ExpertWeights for an expert id.
    shared: the always-active shared expert, or None.
    rows: optional subset of token rows. The expert MLPs and the combine run
      only for these rows. Routing, placement and x quantisation still cover
      all T rows, and the rows left out of y are 0.
    swiglu_limit: clip limit of the SwiGLU (<= 0: no clip).

    Returns a dict with every intermediate:
      ids, w, bitmap, counts, tiles, slot_e/slot_tile/slot_row, rows_of,
      xq, xs, and, indexed by pair id p = t*k + j (shared pairs: T*k + t),
      g, u, h (bf16 bits), hq, hs, o (fp32), plus y (bf16 bits [T][H]).
    """
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    T, H = x_bits.shape
    E = np.asarray(logits).shape[1]
    get = experts if callable(experts) else experts.__getitem__
    out = moe_route(x_bits, logits, k)
    xq, xs = out["xq"], out["xs"]
    n_pairs = T * k + (T if shared is not None else 0)
    I = None
    pair_res = {}

    def run(pair_ids, weights):
        nonlocal I
        toks = np.array([pair_token(p, T, k) for p in pair_ids])
        g, u, h, hq, hs, o = expert_mlp(xq[toks], xs[toks], weights, swiglu_limit)
        I = g.shape[1]
        for n, p in enumerate(pair_ids):
            pair_res[int(p)] = (g[n], u[n], h[n], hq[n], hs[n], o[n])

    for e in range(E):
        pairs = expert_pairs(out, T, k, e, rows)
        if pairs:
            run(pairs, get(e))
    if shared is not None:
        pairs = expert_pairs(out, T, k, "shared", rows)
        if pairs:
            run(pairs, shared)

    y = np.zeros((T, H), dtype=np.uint16)
    if I is not None:
        g_all = np.zeros((n_pairs, I), dtype=np.uint16)
        u_all = np.zeros((n_pairs, I), dtype=np.uint16)
        h_all = np.zeros((n_pairs, I), dtype=np.uint16)
        hq_all = np.zeros((n_pairs, I), dtype=np.uint8)
        hs_all = np.zeros((n_pairs, I // 32), dtype=np.uint8)
        o_all = np.zeros((n_pairs, H), dtype=np.float32)
        for p, (g, u, h, hq, hs, o) in pair_res.items():
            g_all[p], u_all[p], h_all[p], hq_all[p], hs_all[p], o_all[p] = g, u, h, hq, hs, o
        out.update(g=g_all, u=u_all, h=h_all, hq=hq_all, hs=hs_all, o=o_all)
        y = combine(out["w"], o_all, T, k, shared is not None, rows)
    out["y"] = y
    return out
