"""GPU parity with no tolerance, and corner cases of the routing and the combine.

* Exact arithmetic. On structured inputs (synth.exact_case) every binary32
  sum of the step is exact in any order, so g, u, h, their MXFP8 codes, o and
  y are defined bit for bit. Both expert kernels, and MXFP4 weights on the
  tensor-core kernel, must reproduce the oracle exactly. This pins the
  handling of the UE8M0 block scales along K (per 32-group, per weight row
  and per token row) with no tolerance to hide an error. Source: "Beyond
  Day-0: Optimizing DeepSeek-V4.1 Flash in SGLang", 2.1 (group-32 scales,
  Blackwell MXFP8) and 3.1 (the original intermediate rounding).
* A zero combine weight: an expert whose softmax weight underflows to 0
  leaves y independent of that expert's weights.
* Signed zeros among the logits: -0.0 and +0.0 are equal logits and tie to
  the lower expert id ("Routing without sorting" keeps the top-k choices).
* Activation outliers: token rows whose 32-groups span a wide exponent range.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from moe_expert_layer_top_gb300 import abi, synthetic

from gpu_cases import (CudaStep, check_h_close, check_h_quantizer_bit_exact, check_routing_bit_exact,
                       check_xquant_bit_exact, check_y, oracle_abs_sums, oracle_experts, rel_fro, to_np)

pytestmark = pytest.mark.gpu

PATHS = {"gemv": abi.MOE_FLAG_PATH_GEMV, "mma": abi.MOE_FLAG_PATH_MMA}


@pytest.fixture(scope="module", autouse=True)
def built():
    import moe_expert_layer_top_gb300 as pkg
    pkg.build.build()
    abi.load()
    assert torch.cuda.is_available()


# ----------------------------------------------------------------- exact arithmetic

EXACT = [
    # T, routing, shared: one 16-row chunk; 32-row chunks and multi-tile experts; 64-row chunks + shared
    (6, "uniform", 0),
    (40, "zipf", 0),
    (300, "zipf", 1),
]
EXACT_KERNELS = [("mxfp8", "gemv"), ("mxfp8", "mma"), ("mxfp4", "mma")]


def _exact_sums_hold(r, get, sh, T, k):
    """Preconditions of the exact case, on the oracle's side: every gate sum is
    large enough that silu(g) rounds to g in binary32, and every down sum is
    an exact binary32 value whose terms stay within 2^24 of their common unit."""
    assert oracle.bf16_bits_to_f64(r["g"]).min() >= 32.0
    hd = oracle.mxfp8_dequantize(r["hq"], r["hs"])
    x = oracle.mxfp8_dequantize(r["xq"], r["xs"])
    E = len(r["rows_of"])
    for e in list(range(E)) + (["shared"] if sh is not None else []):
        pairs = oracle.expert_pairs(r, T, k, e)
        if not pairs:
            continue
        w = sh if e == "shared" else get(e)
        xt = np.abs(x[[oracle.pair_token(p, T, k) for p in pairs]])
        for name in ("gate", "up"):  # grid values: products are multiples of 2^-8
            wm = w.dequant(name)
            s64 = x[[oracle.pair_token(p, T, k) for p in pairs]] @ wm.T
            np.testing.assert_array_equal(s64.astype(np.float32).astype(np.float64), s64)
            assert (xt @ np.abs(wm).T).max() < 2.0 ** 24 * 2.0 ** -8
        wd = w.dequant("down")
        o64 = hd[pairs] @ wd.T
        np.testing.assert_array_equal(o64.astype(np.float32).astype(np.float64), o64)
        # every partial sum is a multiple of the products' common unit and below 2^24 units:
        # E4M3 values have 3 fraction bits, the grid weights 1 (m in {1, 1.5})
        ah = np.abs(hd[pairs])
        hmin = np.where(ah > 0, ah, np.inf).min(axis=1)
        unit_h = np.where(np.isfinite(hmin), np.exp2(np.floor(np.log2(np.where(np.isfinite(hmin), hmin, 1.0))) - 3),
                          1.0)
        unit_w = np.exp2(np.floor(np.log2(np.abs(wd[wd != 0]).min())) - 1)
        assert np.all((ah @ np.abs(wd).T) < 2.0 ** 24 * (unit_h * unit_w)[:, None])


@pytest.mark.parametrize("fmt,path", EXACT_KERNELS, ids=[f"{f}_{p}" for f, p in EXACT_KERNELS])
@pytest.mark.parametrize("T,routing,shared", EXACT, ids=[f"T{c[0]}_{c[1]}_sh{c[2]}" for c in EXACT])
def test_exact_arithmetic_bit_exact(T, routing, shared, fmt, path):
    H, E, k, I = 512, 8, 2, 256
    c = synth.exact_case(9, T, H, E, k, I, shared, routing)
    w = synthetic.weights_from_bf16(c["gate"], c["up"], c["down"], c.get("sh_gate"), c.get("sh_up"),
                                    c.get("sh_down"), fmt=fmt)
    torch.cuda.synchronize()
    ref_w = [oracle.expert_weights_from_bf16(c["gate"][e], c["up"][e], c["down"][e], fmt) for e in range(E)]
    sh = oracle.expert_weights_from_bf16(c["sh_gate"], c["sh_up"], c["sh_down"], fmt) if shared else None
    for e in (0, E - 1):  # the device's quantisation of the weights is the oracle's, and it is lossless
        np.testing.assert_array_equal(to_np(w.w_gate[e]), ref_w[e].w_gate)
        np.testing.assert_array_equal(to_np(w.s_up[e]), ref_w[e].s_up)
        np.testing.assert_array_equal(to_np(w.w_down[e]), ref_w[e].w_down)
        np.testing.assert_array_equal(ref_w[e].dequant("gate"), oracle.bf16_bits_to_f64(c["gate"][e]))
    g = CudaStep(T, H, E, k, I, shared=shared, weights=w, x_lg=(c["x"], c["logits"]), fmt=fmt,
                 flags=PATHS[path]).run()
    assert g.status_code == abi.MOE_OK, (abi.moe_status_string(g.status_code), g.diag)
    r = oracle.moe_step(c["x"], c["logits"], k, ref_w.__getitem__, shared=sh)
    _exact_sums_hold(r, ref_w.__getitem__, sh, T, k)
    check_routing_bit_exact(g, r)
    check_xquant_bit_exact(g, r)
    np.testing.assert_array_equal(g.t["h_bf16"].view(np.uint16), r["h"])
    np.testing.assert_array_equal(g.t["hq"], r["hq"])
    np.testing.assert_array_equal(g.t["hs"], r["hs"])
    np.testing.assert_array_equal(g.t["o"].view(np.uint32), r["o"].view(np.uint32))
    np.testing.assert_array_equal(g.y_bits, r["y"])
    g.close()


# ----------------------------------------------------------------- zero combine weight

@pytest.mark.parametrize("path", list(PATHS))
def test_zero_weight_expert_leaves_y_unchanged(path):
    """Every row picks expert Z = 5 second, 200 below its first choice: its
    softmax weight underflows to exactly 0. Replacing Z's weights by another
    expert's changes its o, but not one bit of y."""
    T, H, E, k, I, Z = 20, 512, 8, 3, 256, 5
    lg = np.full((T, E), -1000.0, dtype=np.float32)
    for t in range(T):
        a, b = (t % 4), 6 + (t % 2)
        lg[t, a] = 0.0
        lg[t, b] = -1.5
        lg[t, Z] = -200.0
    x = synth.x_bf16(13, T, H)
    w = synthetic.make_weights(13, E, H, I, 0)
    g1 = CudaStep(T, H, E, k, I, weights=w, x_lg=(x, lg), flags=PATHS[path]).run()
    assert g1.status_code == abi.MOE_OK
    assert np.all(g1.t["topk_ids"][:, 2] == Z) and np.all(g1.t["topk_w"][:, 2] == 0.0)
    r = oracle.moe_step(x, lg, k, oracle_experts(13, E, H, I))
    check_routing_bit_exact(g1, r)
    check_y(g1.y_bits, r["y"])
    for name in ("w_gate", "s_gate", "w_up", "s_up", "w_down", "s_down"):
        getattr(w, name)[Z].copy_(getattr(w, name)[Z - 1])
    g2 = CudaStep(T, H, E, k, I, weights=w, x_lg=(x, lg), flags=PATHS[path]).run()
    assert g2.status_code == abi.MOE_OK
    pz = np.arange(T) * k + 2
    assert rel_fro(g2.t["o"][pz], g1.t["o"][pz]) > 0.1        # Z's own output did change
    np.testing.assert_array_equal(g2.y_bits, g1.y_bits)
    g1.close()
    g2.close()


# ----------------------------------------------------------------- signed zeros

def test_signed_zero_logits_tie_to_the_lower_id():
    T, H, E, k, I = 4, 512, 8, 3, 256
    nz, pz = np.float32(-0.0), np.float32(0.0)
    lg = np.full((T, E), -1.0, dtype=np.float32)
    lg[0, :4] = [1.0, 0.5, nz, pz]          # k-th / (k+1)-th boundary: -0 (id 2) against +0 (id 3)
    lg[1, [1, 4, 6]] = [nz, pz, 2.0]        # inside the top-k: -0 (id 1) before +0 (id 4)
    lg[2, :] = [nz, pz, nz, pz, nz, pz, nz, pz]
    lg[3, [0, 7]] = [pz, nz]                # a zero logit first, the other sign last
    x = synth.x_bf16(21, T, H)
    g = CudaStep(T, H, E, k, I, x_lg=(x, lg)).run()
    assert g.status_code == abi.MOE_OK
    r = oracle.moe_step(x, lg, k, oracle_experts(42, E, H, I))
    check_routing_bit_exact(g, r)
    np.testing.assert_array_equal(g.t["topk_ids"][0], [0, 1, 2])
    np.testing.assert_array_equal(g.t["topk_ids"][1], [6, 1, 4])
    np.testing.assert_array_equal(g.t["topk_ids"][2], [0, 1, 2])
    np.testing.assert_array_equal(g.t["topk_ids"][3], [0, 7, 1])
    check_y(g.y_bits, r["y"])
    g.close()


# ----------------------------------------------------------------- activation outliers

@pytest.mark.parametrize("path", list(PATHS))
def test_activation_outliers_parity(path):
    """About one element in 97 of x is 2^4..2^12 times larger: MXFP8 groups of x
    (and of the h they produce) hold values many binades below their maximum."""
    T, H, E, k, I = 40, 512, 8, 2, 256
    x = synth.x_bf16_outliers(17, T, H)
    lg = synth.router_logits(17, T, E, k, "zipf")
    g = CudaStep(T, H, E, k, I, "zipf", 1, seed=17, x_lg=(x, lg), flags=PATHS[path]).run()
    assert g.status_code == abi.MOE_OK
    get = oracle_experts(17, E, H, I)
    sh = oracle.expert_weights_from_synth(17, "shared", H, I)
    r = oracle.moe_step(x, lg, k, get, shared=sh)
    check_routing_bit_exact(g, r)
    check_xquant_bit_exact(g, r)
    check_h_quantizer_bit_exact(g)
    sg, su = oracle_abs_sums(r, T, k, get, sh)
    check_h_close(g, r, np.arange(T * k + T), sg, su)
    check_y(g.y_bits, r["y"])
    g.close()
