"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same seeded inputs, and compare.

Tolerances for the bf16 output y follow the target statement:
* relative Frobenius error <= 1e-2;
* max-abs error <= 5e-2 * rms(y_oracle).
Routing, placement and every MXFP8 quantisation must match bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from moe_expert_layer_top_gb300 import abi, synthetic
from moe_expert_layer_top_gb300.layer import MoEStep, taps_for

Y_REL_FRO = 1e-2
Y_MAX_ABS_RMS = 5e-2


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def bf16_dev_to_bits(t: torch.Tensor) -> np.ndarray:
    return to_np(t.view(torch.int16)).view(np.uint16)


def rel_fro(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a - b))


def check_y(y_gpu_bits, y_ref_bits):
    yg = oracle.bf16_bits_to_f64(y_gpu_bits)
    yr = oracle.bf16_bits_to_f64(y_ref_bits)
    rms = float(np.sqrt(np.mean(yr ** 2)))
    fro = rel_fro(yg, yr)
    mx = float(np.max(np.abs(yg - yr))) if yr.size else 0.0
    assert fro <= Y_REL_FRO, f"relative Frobenius error {fro:.3e}"
    assert mx <= Y_MAX_ABS_RMS * rms, f"max abs error {mx:.3e} vs rms {rms:.3e}"
    return fro, mx, rms


class CudaStep:
    """One CUDA-path step with every tap, on seeded inputs."""

    def __init__(self, T, H, E, k, I, routing="uniform", shared=0, seed=42, weights=None, max_rows=None,
                 flags=0, timeout_ns=0, x_lg=None, fmt="mxfp8", swiglu_limit=0.0):
        self.T, self.H, self.E, self.k, self.I, self.shared, self.seed = T, H, E, k, I, shared, seed
        self.fmt, self.swiglu_limit = fmt, swiglu_limit
        dev = torch.device("cuda", 0)
        self.weights = weights if weights is not None else synthetic.make_weights(seed, E, H, I, shared, dev, fmt)
        if x_lg is None:
            self.x_dev, self.lg_dev, self.x_bits, self.lg = synthetic.make_inputs(seed, T, H, E, k, routing, dev)
        else:
            self.x_bits, self.lg = x_lg
            self.x_dev = torch.from_numpy(self.x_bits.view(np.int16).copy()).view(torch.bfloat16).to(dev)
            self.lg_dev = torch.from_numpy(self.lg.copy()).to(dev)
        self.step = MoEStep(H, I, E, k, self.weights, max_rows or max(T, 1), shared, flags, timeout_ns,
                            weight_format=abi.MOE_WEIGHTS_MXFP4 if fmt == "mxfp4" else abi.MOE_WEIGHTS_MXFP8,
                            swiglu_limit=swiglu_limit)
        self.taps_struct, self.taps = taps_for(T, k, E, H, I, shared, dev)
        self.status = torch.full((1,), -1, dtype=torch.int32, device=dev)

    def run(self):
        y = self.step.forward(self.x_dev, self.lg_dev, taps=self.taps_struct, d_status=self.status)
        torch.cuda.synchronize()
        self.y_bits = bf16_dev_to_bits(y)
        self.t = {n: to_np(v) for n, v in self.taps.items()}
        self.status_code = int(self.status.item())
        self.diag = self.step.diagnostics() if self.status_code != abi.MOE_OK else None
        return self

    def close(self):
        self.step.close()


def oracle_experts(seed, E, H, I, cache=None, fmt="mxfp8"):
    cache = {} if cache is None else cache

    def get(e):
        key = (seed, e, H, I, fmt)
        if key not in cache:
            cache[key] = oracle.expert_weights_from_synth(seed, e, H, I, fmt=fmt)
        return cache[key]
    return get


def check_routing_bit_exact(g: CudaStep, r: dict):
    np.testing.assert_array_equal(g.t["topk_ids"], r["ids"])
    np.testing.assert_array_equal(g.t["topk_w"].view(np.uint32), r["w"].view(np.uint32))
    np.testing.assert_array_equal(g.t["bitmap"].view(np.uint32), r["bitmap"])
    np.testing.assert_array_equal(g.t["counts"], r["counts"])
    ref_slot = (r["slot_e"].astype(np.int64) << 16) | (r["slot_tile"] * 8 + r["slot_row"])
    np.testing.assert_array_equal(g.t["slot"].astype(np.int64), ref_slot)


def check_xquant_bit_exact(g: CudaStep, r: dict):
    np.testing.assert_array_equal(g.t["xq"], r["xq"])
    np.testing.assert_array_equal(g.t["xs"], r["xs"])


def check_h_quantizer_bit_exact(g: CudaStep, pairs=None):
    """The GPU's MXFP8 h must be the oracle's quantisation of the GPU's own bf16 h."""
    hb = g.t["h_bf16"].view(np.uint16)
    if pairs is not None:
        hb = hb[pairs]
    q, s = oracle.mxfp8_quantize(oracle.bf16_bits_to_f64(hb))
    hq, hs = g.t["hq"], g.t["hs"]
    if pairs is not None:
        hq, hs = hq[pairs], hs[pairs]
    np.testing.assert_array_equal(hq, q)
    np.testing.assert_array_equal(hs, s)


def bf16_step(v) -> np.ndarray:
    """Spacing of bf16 values at |v| (one unit in the last place; subnormal spacing below 2^-126)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


SILU_MIN_AT = -1.2784645427610738   # the one stationary point of silu(g) = g sigmoid(g)


def _silu(g):
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def h_envelope(g_bits, u_bits, sum_g, sum_u, K_gate: int, lim: float = 0.0):
    """Bounds [lo, hi] for the device's bf16 h = bf16(silu(g') u'), derived from
    the arithmetic, given the oracle's g and u (bf16 bits, rounded from the
    exact sums) and sum_k |x_k w_k| of each.

    The device sums K_gate products in binary32 in its own order: its sum is
    within K_gate * 2^-24 * sum|x w| of the exact one (the recursive-summation
    bound), and its bf16 g' within that plus one bf16 step of the oracle's g.
    The same holds for u'. h = silu(min(g', L)) * clamp(u', -L, L) is taken
    at the ends of both intervals (and at silu's stationary point when it lies
    inside), and the result may round by one more bf16 step each way.
    The device evaluates silu(g) = g / (1 + exp(-g)) in binary32, where exp(-g)
    overflows for g < -88.72 and silu(g) becomes -0; there the exact value has
    magnitude below 88.73 e^-88.72 < 2^-121, so h may also be off by up to
    |u'| 2^-121 (a value below 1e-36 where it matters at all)."""
    gb = oracle.bf16_bits_to_f64(np.asarray(g_bits, dtype=np.uint16))
    ub = oracle.bf16_bits_to_f64(np.asarray(u_bits, dtype=np.uint16))
    eps = K_gate * 2.0 ** -24
    dg = bf16_step(gb) + eps * sum_g
    du = bf16_step(ub) + eps * sum_u
    gs = [gb - dg, gb, gb + dg]
    inside = (gb - dg < SILU_MIN_AT) & (gb + dg > SILU_MIN_AT)
    gs.append(np.where(inside, SILU_MIN_AT, gb))
    us = [ub - du, ub + du]
    if lim > 0:
        L = float(np.float32(lim))
        gs = [np.minimum(g, L) for g in gs]
        us = [np.clip(u, -L, L) for u in us]
    vals = [_silu(g) * u for g in gs for u in us]
    lo = np.minimum.reduce(vals)
    hi = np.maximum.reduce(vals)
    tail = np.maximum.reduce([np.abs(u) for u in us]) * 2.0 ** -121
    lo = lo - bf16_step(lo) - tail
    hi = hi + bf16_step(hi) + tail
    return lo, hi


def check_h_close(g: CudaStep, r: dict, pairs, sum_g, sum_u, lim: float = 0.0):
    """bf16 h: every value inside the envelope that one-step flips of g and u
    and the device's fp32 accumulation allow (h_envelope). Returns the
    fraction of h values that differ from the oracle's at all."""
    pairs = np.asarray(pairs)
    hg = g.t["h_bf16"].view(np.uint16)[pairs]
    hr = r["h"][pairs]
    lo, hi = h_envelope(r["g"][pairs], r["u"][pairs], sum_g[pairs], sum_u[pairs], g.H, lim)
    v = oracle.bf16_bits_to_f64(hg)
    bad = ~((v >= lo) & (v <= hi))
    if np.any(bad):
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{int(bad.sum())} h values outside the envelope; first pair {pairs[i[0]]} column "
                             f"{i[1]}: {v[tuple(i)]!r} not in [{lo[tuple(i)]!r}, {hi[tuple(i)]!r}], "
                             f"oracle {oracle.bf16_bits_to_f64(hr[tuple(i)])!r}")
    return float(np.mean(hg != hr))


def oracle_abs_sums(r: dict, T: int, k: int, get, shared_w=None):
    """sum_k |x_k w_k| of the gate and up projections for every pair [P][I],
    from the oracle's dequantised token rows and weights (for h_envelope)."""
    x = np.abs(oracle.mxfp8_dequantize(r["xq"], r["xs"]))
    P, I = r["h"].shape
    sg = np.zeros((P, I))
    su = np.zeros((P, I))
    E = len(r["rows_of"])
    for e in list(range(E)) + (["shared"] if shared_w is not None else []):
        pairs = oracle.expert_pairs(r, T, k, e)
        if not pairs:
            continue
        w = shared_w if e == "shared" else get(e)
        toks = [oracle.pair_token(p, T, k) for p in pairs]
        sg[pairs] = x[toks] @ np.abs(w.dequant("gate")).T
        su[pairs] = x[toks] @ np.abs(w.dequant("up")).T
    return sg, su


def full_oracle(seed: int, steps: dict, H: int, I: int, fmt: str = "mxfp8", lim: float = 0.0):
    """The oracle over every token row of several steps that share one set of
    seeded expert weights: steps = {tag: (x_bits, logits, k, shared)}. The
    expert MLPs run in a spawn pool, one expert per task (oracle_pool).
    Returns ({tag: result dict as oracle.moe_step gives, plus sum_g and sum_u},
    {expert: sha256 of each of its quantised weight tensors})."""
    import oracle_pool
    routes = {}
    jobs = {}
    for tag, (x_bits, lg, k, shared) in steps.items():
        T = x_bits.shape[0]
        rt = oracle.moe_route(x_bits, lg, k)
        routes[tag] = rt
        E = lg.shape[1]
        for e in list(range(E)) + (["shared"] if shared else []):
            pairs = oracle.expert_pairs(rt, T, k, e)
            if pairs:
                toks = [oracle.pair_token(p, T, k) for p in pairs]
                jobs.setdefault(e, []).append((tag, rt["xq"][toks], rt["xs"][toks]))
    tasks = [(seed, e, H, I, fmt, lim, j) for e, j in jobs.items()]
    res, hashes = oracle_pool.run_experts(tasks)
    out = {}
    for tag, (x_bits, lg, k, shared) in steps.items():
        rt = routes[tag]
        T = x_bits.shape[0]
        P = T * k + (T if shared else 0)
        arrs = {"g": np.zeros((P, I), np.uint16), "u": np.zeros((P, I), np.uint16),
                "h": np.zeros((P, I), np.uint16), "hq": np.zeros((P, I), np.uint8),
                "hs": np.zeros((P, I // 32), np.uint8), "o": np.zeros((P, H), np.float32),
                "sum_g": np.zeros((P, I)), "sum_u": np.zeros((P, I))}
        for e in res:
            if tag not in res[e]:
                continue
            pairs = oracle.expert_pairs(rt, T, k, e)
            for name, v in zip(("g", "u", "h", "hq", "hs", "o", "sum_g", "sum_u"), res[e][tag]):
                arrs[name][pairs] = v
        rt = dict(rt)
        rt.update(arrs)
        rt["y"] = oracle.combine(rt["w"], arrs["o"], T, k, shared)
        out[tag] = rt
    return out, hashes
