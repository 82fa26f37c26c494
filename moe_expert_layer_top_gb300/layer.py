"""PyTorch-facing wrapper of the C ABI: device tensors in, device tensors out.

PyTorch only supplies device memory and streams here. Every step of the MoE
computation runs in libmoe.so. If the library cannot be loaded, or a call
fails, this raises; there is no fallback.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import abi


@dataclass
class MoEWeightsMXFP8:
    """Canonical expert weights on the device (uint8 tensors).

    MXFP8: w_gate, w_up: [E][I][H] E4M3;  s_gate, s_up: [E][I][H/32] UE8M0
           w_down:       [E][H][I] E4M3;  s_down:       [E][H][I/32] UE8M0
    MXFP4: the same with w_gate, w_up [E][I][H/2] and w_down [E][H][I/2] of
           packed E2M1 codes (element 2i in the low nibble).
    sh_*: the same for one shared expert without the E axis, or None.
    """
    w_gate: torch.Tensor
    s_gate: torch.Tensor
    w_up: torch.Tensor
    s_up: torch.Tensor
    w_down: torch.Tensor
    s_down: torch.Tensor
    sh_w_gate: torch.Tensor | None = None
    sh_s_gate: torch.Tensor | None = None
    sh_w_up: torch.Tensor | None = None
    sh_s_up: torch.Tensor | None = None
    sh_w_down: torch.Tensor | None = None
    sh_s_down: torch.Tensor | None = None

    def as_abi(self) -> abi.MoeWeights:
        w = abi.MoeWeights()
        for name, _ in abi.MoeWeights._fields_:
            setattr(w, name, abi.ptr(getattr(self, name)))
        return w


def quantize_mxfp4(x: torch.Tensor, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """MXFP4 (E2M1 packed two per byte, group-32 UE8M0) quantisation of bf16 rows along the last axis."""
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA bf16 tensor")
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    q = torch.empty(x.shape[:-1] + (cols // 2,), dtype=torch.uint8, device=x.device)
    s = torch.empty(x.shape[:-1] + (cols // 32,), dtype=torch.uint8, device=x.device)
    st = stream if stream is not None else torch.cuda.current_stream(x.device)
    abi.check("moe_quantize_mxfp4", abi.moe_quantize_mxfp4(x, rows, cols, q, s, st))
    return q, s


def quantize_mxfp8(x: torch.Tensor, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """MXFP8 (E4M3, group-32 UE8M0) quantisation of bf16 rows along the last axis, on the device."""
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA bf16 tensor")
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    s = torch.empty(x.shape[:-1] + (cols // 32,), dtype=torch.uint8, device=x.device)
    st = stream if stream is not None else torch.cuda.current_stream(x.device)
    abi.check("moe_quantize_mxfp8", abi.moe_quantize_mxfp8(x, rows, cols, q, s, st))
    return q, s


class MoEStep:
    """One planned MoE layer (Guard + Build at construction, Runtime per forward)."""

    def __init__(self, hidden: int, intermediate: int, num_experts: int, top_k: int, weights: MoEWeightsMXFP8,
                 max_rows: int, num_shared: int = 0, flags: int = 0, wait_timeout_ns: int = 0, stream=None,
                 weight_format: int = 0, swiglu_limit: float = 0.0):
        self.cfg = abi.MoeConfig(hidden, intermediate, num_experts, top_k, num_shared, max_rows, flags,
                                 wait_timeout_ns, weight_format, swiglu_limit)
        self.weights = weights  # keeps the device buffers alive for the plan's lifetime
        self.H, self.I, self.E, self.k, self.shared = hidden, intermediate, num_experts, top_k, num_shared
        self.max_rows = max_rows
        self.plan = abi.moe_plan(self.cfg, weights.as_abi(), stream)

    def forward(self, x: torch.Tensor, logits: torch.Tensor, y: torch.Tensor | None = None,
                taps: abi.MoeTaps | None = None, d_status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, self.H), dtype=torch.bfloat16, device=x.device)
        st = stream if stream is not None else torch.cuda.current_stream(x.device)
        abi.check("moe_forward", abi.moe_forward(self.plan, x, logits, T, y, taps, d_status, st))
        return y

    def forward_dev(self, x: torch.Tensor, logits: torch.Tensor, d_T: torch.Tensor, y: torch.Tensor,
                    d_status: torch.Tensor | None = None, stream=None) -> None:
        """A step whose row count is read on the device from d_T (int32, one element):
        capture it once in a CUDA graph and replay it for any T <= max_rows.
        x, logits and y hold max_rows rows; rows at or past T are not touched."""
        st = stream if stream is not None else torch.cuda.current_stream(x.device)
        abi.check("moe_forward_dev", abi.moe_forward_dev(self.plan, x, logits, d_T, y, d_status, st))

    def forward_fused(self, x: torch.Tensor, w_router: torch.Tensor | None = None,
                      logits: torch.Tensor | None = None, resid: torch.Tensor | None = None,
                      norm_weight: torch.Tensor | None = None, rms_eps: float = 1e-6,
                      mix_res: torch.Tensor | None = None, mix_post: torch.Tensor | None = None,
                      mix_pre: torch.Tensor | None = None, in_place: bool = False, z_tap: bool = False,
                      taps: abi.MoeTaps | None = None, d_status: torch.Tensor | None = None,
                      stream=None) -> dict:
        """One step with the steps on either side fused into its kernels.

        w_router (bf16 [E][H]) computes the logits on the device; they are
        returned as "logits". Without it, logits (fp32 [T][E]) is the input.
        resid (bf16 [T][S][H], S <= 4) turns on the epilogue. It returns the
        new streams ("resid", the same tensor when in_place) and the next
        layer's MXFP8 input ("zq", "zs"), plus "z" (bf16) when z_tap is set.
        """
        T = x.shape[0]
        dev = x.device
        out = {"y": torch.empty((T, self.H), dtype=torch.bfloat16, device=dev)}
        if w_router is not None:
            out["logits"] = logits if logits is not None else torch.empty((T, self.E), dtype=torch.float32,
                                                                             device=dev)
        io = abi.fused_io(w_router=w_router, logits=out.get("logits", logits))
        if resid is not None:
            S = resid.shape[1]
            out["resid"] = resid if in_place else torch.empty_like(resid)
            out["zq"] = torch.empty((T, self.H), dtype=torch.uint8, device=dev)
            out["zs"] = torch.empty((T, self.H // 32), dtype=torch.uint8, device=dev)
            if z_tap:
                out["z"] = torch.empty((T, self.H), dtype=torch.bfloat16, device=dev)
            io = abi.fused_io(w_router=w_router, logits=out.get("logits", logits), num_streams=S, resid_in=resid,
                              resid_out=out["resid"], mix_res=mix_res, mix_post=mix_post, mix_pre=mix_pre,
                              norm_weight=norm_weight, rms_eps=rms_eps, zq=out["zq"], zs=out["zs"],
                              z=out.get("z"))
        st = stream if stream is not None else torch.cuda.current_stream(dev)
        abi.check("moe_forward_fused", abi.moe_forward_fused(self.plan, x, T, io, out["y"], taps, d_status, st))
        return out

    def forward_host(self, x_host: torch.Tensor, logits_host: torch.Tensor, y_host: torch.Tensor, stream=None) -> int:
        st = stream if stream is not None else torch.cuda.current_stream()
        return abi.moe_forward_host(self.plan, x_host, logits_host, x_host.shape[0], y_host, st)

    def kernel_times(self) -> tuple[float, int]:
        return abi.moe_kernel_times(self.plan)

    def status(self) -> int:
        return abi.moe_plan_status(self.plan)

    def diagnostics(self) -> list[int]:
        return abi.moe_plan_diagnostics(self.plan)

    def close(self):
        if self.plan:
            abi.moe_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def taps_for(T: int, k: int, E: int, H: int, I: int, shared: int, device) -> tuple[abi.MoeTaps, dict]:
    """Allocate every debug tap for a T-row step. Returns (struct, dict of tensors)."""
    P = T * k + T * shared
    words = (T + 31) // 32
    t = {
        "topk_ids": torch.empty((T, k), dtype=torch.int32, device=device),
        "topk_w": torch.empty((T, k), dtype=torch.float32, device=device),
        "bitmap": torch.empty((E, words), dtype=torch.int32, device=device),
        "counts": torch.empty((E,), dtype=torch.int32, device=device),
        "slot": torch.empty((T, k), dtype=torch.int32, device=device),
        "xq": torch.empty((T, H), dtype=torch.uint8, device=device),
        "xs": torch.empty((T, H // 32), dtype=torch.uint8, device=device),
        "h_bf16": torch.empty((P, I), dtype=torch.int16, device=device),
        "hq": torch.empty((P, I), dtype=torch.uint8, device=device),
        "hs": torch.empty((P, I // 32), dtype=torch.uint8, device=device),
        "o": torch.empty((P, H), dtype=torch.float32, device=device),
    }
    s = abi.MoeTaps()
    for name, _ in abi.MoeTaps._fields_:
        setattr(s, name, abi.ptr(t[name]))
    return s, t
