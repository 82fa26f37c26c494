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


def check_h_close(g: CudaStep, r: dict, pairs):
    """bf16 h: equal except for rare one-ulp rounding flips."""
    hg = g.t["h_bf16"].view(np.uint16)[pairs].astype(np.int32)
    hr = r["h"][pairs].astype(np.int32)
    diff = np.abs(hg - hr)
    frac = float(np.mean(diff != 0))
    assert frac <= 1e-2, f"{frac:.2%} of h differ"
    assert rel_fro(oracle.bf16_bits_to_f64(hg.astype(np.uint16)), oracle.bf16_bits_to_f64(hr.astype(np.uint16))) <= 1e-2
    return frac
