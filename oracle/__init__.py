"""CPU oracle for the small-batch MXFP8 MoE step. TEST INFRASTRUCTURE ONLY.

A plain, slow and obviously correct restatement of the decode MoE step, in
numpy. Floating-point work is in fp64 unless the method fixes a narrower
type. Its users are ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline of ``bench.py``. Nothing in the product path imports it, and it
imports nothing from the product package. It shares no code with the CUDA
path. The only thing both sides take from one place is the seeded input
generator in ``synth/``, which holds none of the method's arithmetic.

Sources, cited by page title and section:

* "SGLang's Low-Latency Mode Boosts DeepSeek-V4.1-Flash Speed by 1.56x on AMD",
  section "NVIDIA overlaps the dependency chain", bullet "Routing without
  sorting". Each expert's token rows are placed into 8-row tiles using a
  per-expert bitmap and population counts, with no scan or sort, and the
  top-k choices are kept.
* "Beyond Day-0: Optimizing DeepSeek-V4.1 Flash in SGLang", section 2.1:
  - group-32 FP8 weights with scales in the Blackwell MXFP8 layout;
  - MXFP8 quantisation fused into the producers of activations;
  - the router emits the downstream layout;
  - the weighted reduction of expert outputs is fused with the
    shared-expert addition.
* The same page, section 3.1. The MoE kernels fuse the clipped SwiGLU and
  keep the original intermediate rounding.
* "FlyDSL Mono Kernels for High-Interactivity LLM Serving in ATOM", section
  "MiniMax-M3: Connecting Attention and Experts". Each expert does its
  up/gate and down projections, for the shared and the routed experts.
* "Beyond Day-0 ...", section 2.1, the MoE, mHC and small-operator bullets:
  the router projection in front of the step, and behind it the residual-stream
  combination, the next layer's input combination, RMSNorm and MXFP8
  quantisation (``oracle/fused.py``).
* OCP Microscaling Formats (MX) Specification v1.0:
  - the E4M3 and E2M1 element encodings (MXFP8, MXFP4);
  - the UE8M0 scale;
  - the rule for choosing a group's shared scale.

Readings where the pages are silent are stated in each function's docstring.
All of these functions are pinned by ``tests/test_oracle_*.py``. Pins include
brute force, closed forms, hand-worked examples in ``tests/golden/`` and
special cases that reduce to textbook routines.
"""
from .formats import (  # noqa: F401
    E2M1_MAX,
    E4M3_MAX,
    bf16_bits_to_f64,
    e2m1_decode,
    e2m1_encode,
    e4m3_decode,
    e4m3_encode,
    f32_to_bf16_bits,
    mxfp4_dequantize,
    mxfp4_quantize,
    mxfp8_dequantize,
    mxfp8_quantize,
    pack_e2m1,
    ue8m0_value,
    unpack_e2m1,
)
from .fused import residual_norm_mxfp8, router_logits  # noqa: F401
from .routing import exp_rn, placement, softmax_topk_weights, topk_ids  # noqa: F401
from .step import (ExpertWeights, combine, expert_mlp, expert_pairs, expert_weights_from_bf16,  # noqa: F401
                   expert_weights_from_synth, moe_route, moe_step, pair_token)
