"""The steps on either side of the MoE step.

In front: the router projection, logits = x . W_r^T.
Behind: the residual-stream combination, the next layer's input
combination, RMSNorm, and MXFP8 quantisation of the normalised row.

Oracle module (test infrastructure only). See ``oracle/__init__.py``.

Passages followed ("Beyond Day-0: Optimizing DeepSeek-V4.1 Flash in SGLang",
section 2.1):

* The MoE bullet. The router produces the layout that downstream computation
  needs. Where supported, the kernels also fuse the mHC output combination,
  the next layer's input combination, or normalisation, to cut intermediate
  writes to GPU memory.
* The mHC bullet. The weighted combination of mHC's four residual streams is
  fused with RMSNorm, with quantisation added on supported paths.
* The small-operator bullet. Q RMSNorm is fused with MXFP8 quantisation.

Readings where the pages are silent:

* Router projection. x (bf16) times W_r (bf16, [E][H], one row per routed
  expert), with no bias and no scaling. Every product of two bf16 values is
  exact in fp64, and the sum over H is an fp64 matrix product (a library
  primitive). The logits are rounded once to fp32, the type the device
  accumulates in and the type the top-k reads.
* Residual streams. Each token row carries S residual streams (S = 1 is the
  plain residual; mHC uses S = 4). Three per-row coefficient sets are inputs
  to the step, computed elsewhere:
  - res [T][S][S], the stream mixing matrix;
  - post [T][S], the weight of the MoE output in each stream;
  - pre [T][S], the next layer's input combination.
  The step does not compute them: the pages compute the mixing coefficients
  on a separate stream and synchronise when the combination needs them.
  Missing sets default to the plain residual: res = identity, post = 1,
  pre = 1.
* Output combination: new_s = sum_s' res[s][s'] * stream_s' + post[s] * y.
  y is the MoE output after its bf16 rounding; new_s is rounded to bf16, the
  stream's storage type. The value is computed in fp64, then rounded to fp32
  and then to bf16.
* Input combination: u = sum_s pre[s] * new_s, held in fp32.
* RMSNorm: z = u * gamma / sqrt(mean_h(u^2) + eps). gamma is bf16 [H] and eps
  is a binary32 value. z is rounded to fp32 and then to bf16.
* z is quantised to MXFP8 along H (groups of 32), by the rule used for x.
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_bits_to_f64, f32_to_bf16_bits, mxfp8_quantize


def router_logits(x_bits, wr_bits) -> np.ndarray:
    """Router logits fp32 [T][E] from x (bf16 bits [T][H]) and W_r (bf16 bits [E][H])."""
    x = bf16_bits_to_f64(np.asarray(x_bits, dtype=np.uint16))
    w = bf16_bits_to_f64(np.asarray(wr_bits, dtype=np.uint16))
    if x.shape[1] != w.shape[1]:
        raise ValueError("x and W_r disagree on H")
    return (x @ w.T).astype(np.float32)


def _coefficients(T: int, S: int, res, post, pre):
    res64 = np.broadcast_to(np.eye(S), (T, S, S)) if res is None else \
        np.asarray(res, dtype=np.float32).astype(np.float64).reshape(T, S, S)
    post64 = np.ones((T, S)) if post is None else np.asarray(post, dtype=np.float32).astype(np.float64).reshape(T, S)
    pre64 = np.ones((T, S)) if pre is None else np.asarray(pre, dtype=np.float32).astype(np.float64).reshape(T, S)
    return res64, post64, pre64


def residual_norm_mxfp8(y_bits, resid_bits, gamma_bits, eps: float, res=None, post=None, pre=None):
    """The fused epilogue over T token rows with S residual streams.

    y_bits: the MoE output, bf16 bits [T][H].
    resid_bits: the residual streams before this layer's output, bf16 bits [T][S][H].
    gamma_bits: RMSNorm weight, bf16 bits [H].
    eps: RMSNorm epsilon (taken as binary32).
    res, post, pre: fp32 coefficient sets [T][S][S], [T][S] and [T][S], or None.

    Returns a dict:
      resid: the new residual streams, bf16 bits [T][S][H];
      u:     the next layer's input combination, fp32 [T][H];
      z32:   the normalised row before its bf16 rounding, fp32 [T][H];
      z:     the normalised row, bf16 bits [T][H];
      zq, zs: z quantised to MXFP8 (E4M3 [T][H], UE8M0 [T][H/32]).
    """
    y = bf16_bits_to_f64(np.asarray(y_bits, dtype=np.uint16))
    r = bf16_bits_to_f64(np.asarray(resid_bits, dtype=np.uint16))
    T, S, H = r.shape
    if y.shape != (T, H):
        raise ValueError("y and the residual streams disagree on shape")
    res64, post64, pre64 = _coefficients(T, S, res, post, pre)
    g = bf16_bits_to_f64(np.asarray(gamma_bits, dtype=np.uint16)).reshape(H)
    eps64 = float(np.float32(eps))

    # output combination: each new stream mixes the old ones and adds the weighted MoE output
    new = np.einsum("tab,tbh->tah", res64, r) + post64[:, :, None] * y[:, None, :]
    new_bits = f32_to_bf16_bits(new.astype(np.float32))
    newf = bf16_bits_to_f64(new_bits)
    # the next layer's input combination, kept in binary32
    u = np.einsum("ts,tsh->th", pre64, newf).astype(np.float32)
    u64 = u.astype(np.float64)
    # RMSNorm over H
    ms = np.mean(u64 * u64, axis=1)
    z32 = (u64 * g[None, :] / np.sqrt(ms + eps64)[:, None]).astype(np.float32)
    z_bits = f32_to_bf16_bits(z32)
    zq, zs = mxfp8_quantize(bf16_bits_to_f64(z_bits))
    return {"resid": new_bits, "u": u, "z32": z32, "z": z_bits, "zq": zq, "zs": zs}
