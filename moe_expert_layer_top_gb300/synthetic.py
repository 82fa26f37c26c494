"""Synthetic MXFP8 / MXFP4 checkpoints and inputs on the device, for tests and benchmarks.

Weights are drawn as bf16 on the device by the seeded generator (synth.gpu),
in chunks of experts. They are then quantised to canonical MXFP8 (or MXFP4)
with this library's own moe_quantize_mxfp8 (moe_quantize_mxfp4), as a user
would quantise a bf16 checkpoint. The oracle draws the same bf16 values on
the host and quantises them with its own rules, so nothing computed here
feeds the oracle.
Token rows and router logits are small and are drawn on the host
(synth.x_bf16, synth.router_logits), then copied to the device.
"""
from __future__ import annotations

import numpy as np
import torch

import synth
import synth.gpu

from .layer import MoEWeightsMXFP8, quantize_mxfp4, quantize_mxfp8


def _fill_matrix(seed: int, stream_id: int, rows: int, cols: int, q_out: torch.Tensor, s_out: torch.Tensor,
                 scratch: torch.Tensor, fmt: str):
    """Draw one [rows][cols] bf16 matrix (sigma = 1/sqrt(cols)) and quantise it into q_out/s_out."""
    n = rows * cols
    buf = scratch[:n]
    st = torch.cuda.current_stream()
    synth.gpu.normal_bf16(seed, stream_id, 0, n, synth.expert_sigma(cols), buf.data_ptr(), st.cuda_stream)
    quant = quantize_mxfp4 if fmt == "mxfp4" else quantize_mxfp8
    q, s = quant(buf.view(torch.bfloat16).view(rows, cols))
    q_out.copy_(q)
    s_out.copy_(s)


def make_weights(seed: int, E: int, H: int, I: int, shared: int = 0, device="cuda",
                 fmt: str = "mxfp8") -> MoEWeightsMXFP8:
    """All experts' weights (plus the shared expert's), drawn and quantised on the device.
    fmt "mxfp4" packs two E2M1 codes per byte: w_gate/w_up are [E][I][H/2], w_down [E][H][I/2]."""
    u8 = dict(dtype=torch.uint8, device=device)
    div = 2 if fmt == "mxfp4" else 1
    w = MoEWeightsMXFP8(
        w_gate=torch.empty((E, I, H // div), **u8), s_gate=torch.empty((E, I, H // 32), **u8),
        w_up=torch.empty((E, I, H // div), **u8), s_up=torch.empty((E, I, H // 32), **u8),
        w_down=torch.empty((E, H, I // div), **u8), s_down=torch.empty((E, H, I // 32), **u8))
    scratch = torch.empty((I * H,), dtype=torch.int16, device=device)
    for e in range(E):
        _fill_matrix(seed, synth.stream_gate(e), I, H, w.w_gate[e], w.s_gate[e], scratch, fmt)
        _fill_matrix(seed, synth.stream_up(e), I, H, w.w_up[e], w.s_up[e], scratch, fmt)
        _fill_matrix(seed, synth.stream_down(e), H, I, w.w_down[e], w.s_down[e], scratch, fmt)
    if shared:
        w.sh_w_gate, w.sh_s_gate = torch.empty((I, H // div), **u8), torch.empty((I, H // 32), **u8)
        w.sh_w_up, w.sh_s_up = torch.empty((I, H // div), **u8), torch.empty((I, H // 32), **u8)
        w.sh_w_down, w.sh_s_down = torch.empty((H, I // div), **u8), torch.empty((H, I // 32), **u8)
        _fill_matrix(seed, synth.STREAM_SH_GATE, I, H, w.sh_w_gate, w.sh_s_gate, scratch, fmt)
        _fill_matrix(seed, synth.STREAM_SH_UP, I, H, w.sh_w_up, w.sh_s_up, scratch, fmt)
        _fill_matrix(seed, synth.STREAM_SH_DOWN, H, I, w.sh_w_down, w.sh_s_down, scratch, fmt)
    del scratch
    return w


def make_inputs(seed: int, T: int, H: int, E: int, k: int, routing: str, device="cuda"):
    """Host-drawn token rows (bf16) and router logits (fp32), copied to the device.

    Returns (x_dev bf16 [T][H], logits_dev fp32 [T][E], x_bits numpy uint16, logits numpy fp32)."""
    x_bits = synth.x_bf16(seed, T, H)
    lg = synth.router_logits(seed, T, E, k, routing)
    x_dev = torch.from_numpy(x_bits.view(np.int16).copy()).view(torch.bfloat16).to(device)
    lg_dev = torch.from_numpy(lg.copy()).to(device)
    return x_dev, lg_dev, x_bits, lg


def weights_from_bf16(gate: np.ndarray, up: np.ndarray, down: np.ndarray, sh_gate=None, sh_up=None, sh_down=None,
                      device="cuda", fmt: str = "mxfp8") -> MoEWeightsMXFP8:
    """Canonical weights from given bf16 bit patterns (host uint16 arrays:
    gate, up [E][I][H], down [E][H][I]; sh_* without the E axis), uploaded and
    quantised with this library's moe_quantize_mxfp8 (or _mxfp4)."""
    quant = quantize_mxfp4 if fmt == "mxfp4" else quantize_mxfp8

    def q(bits):
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)
        return quant(t)
    wg, sg = q(gate)
    wu, su = q(up)
    wd, sd = q(down)
    w = MoEWeightsMXFP8(wg, sg, wu, su, wd, sd)
    if sh_gate is not None:
        w.sh_w_gate, w.sh_s_gate = q(sh_gate)
        w.sh_w_up, w.sh_s_up = q(sh_up)
        w.sh_w_down, w.sh_s_down = q(sh_down)
    return w
