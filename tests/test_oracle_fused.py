"""Pins for the oracle's steps either side of the MoE step: the router
projection in front, and the residual-stream combination + RMSNorm + MXFP8
epilogue behind.

The oracle is checked against things that are not itself:
* exact rational sums (fractions.Fraction) of bf16 products, rounded once to fp32;
* one-hot token rows, which select one column of the router weight;
* hand-worked examples in tests/golden/residual_norm_examples.json;
* torch.nn.functional.rms_norm in fp64 (a library routine);
* special cases that reduce to a plain bf16 addition, or to one stream;
* scale invariance of RMSNorm with eps = 0.
Source: "Beyond Day-0: Optimizing DeepSeek-V4.1 Flash in SGLang", section 2.1
(the MoE, mHC and small-operator bullets).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import fused

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits_of(v) -> np.ndarray:
    """bf16 bits of values that are exact in bf16 (checked)."""
    v = np.asarray(v, dtype=np.float32)
    b = (v.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    assert np.array_equal(oracle.bf16_bits_to_f64(b), v.astype(np.float64)), "not exact in bf16"
    return b


# --------------------------------------------------------------------------- router projection

def test_router_logits_equal_exact_rational_sums():
    rng = np.random.default_rng(5)
    T, E, H = 3, 5, 24
    # bf16 values of a limited exponent range, so each exact sum is an fp64 value
    x = (rng.integers(-255, 256, (T, H)) * 2.0 ** rng.integers(-6, 2, (T, H))).astype(np.float32)
    w = (rng.integers(-255, 256, (E, H)) * 2.0 ** rng.integers(-9, -1, (E, H))).astype(np.float32)
    xb, wb = bits_of(x), bits_of(w)
    got = fused.router_logits(xb, wb)
    for t in range(T):
        for e in range(E):
            exact = sum(Fraction(float(x[t, h])) * Fraction(float(w[e, h])) for h in range(H))
            assert Fraction(float(exact)) == exact      # representable in fp64: one rounding below
            assert got[t, e] == np.float32(float(exact)), (t, e)


def test_router_logits_one_hot_rows_select_a_column():
    E, H = 6, 64
    wb = synth.router_weight_bf16(3, E, H)
    cols = [0, 17, 63, 5]
    x = np.zeros((len(cols), H), dtype=np.float32)
    for t, h in enumerate(cols):
        x[t, h] = 1.0
    got = fused.router_logits(bits_of(x), wb)
    w = oracle.bf16_bits_to_f64(wb)
    for t, h in enumerate(cols):
        np.testing.assert_array_equal(got[t], w[:, h].astype(np.float32))


def test_router_logits_permuting_experts_permutes_columns():
    T, E, H = 4, 8, 96
    xb = synth.x_bf16(2, T, H)
    wb = synth.router_weight_bf16(2, E, H)
    perm = np.array([3, 0, 7, 1, 6, 2, 5, 4])
    np.testing.assert_array_equal(fused.router_logits(xb, wb[perm]), fused.router_logits(xb, wb)[:, perm])


def test_router_logits_shape_check():
    with pytest.raises(ValueError):
        fused.router_logits(np.zeros((2, 32), np.uint16), np.zeros((4, 64), np.uint16))


# --------------------------------------------------------------------------- epilogue

def _row(pattern, H=32):
    kind, v = pattern
    if kind == "const":
        return np.full(H, v, dtype=np.float32)
    assert kind == "alt"
    return np.where(np.arange(H) % 2 == 0, v, -v).astype(np.float32)


def _golden_cases():
    with open(os.path.join(GOLDEN, "residual_norm_examples.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"].split()[0])
def test_epilogue_hand_worked_examples(case):
    S, H = case["S"], 32
    streams = np.stack([_row(p) for p in case["streams"]])[None]      # [1][S][H]
    y = _row(case["y"])[None]
    assert streams.shape == (1, S, H)
    coef = {}
    for name in ("res", "post", "pre"):
        coef[name] = None if case[name] is None else np.asarray(case[name], dtype=np.float32)[None]
    gamma = np.full(H, case["gamma"], dtype=np.float32)
    r = fused.residual_norm_mxfp8(bits_of(y), bits_of(streams), bits_of(gamma), case["eps"], **coef)
    for s, p in enumerate(case["expect_resid"]):
        np.testing.assert_array_equal(oracle.bf16_bits_to_f64(r["resid"][0, s]), _row(p))
    np.testing.assert_array_equal(r["u"][0], _row(case["expect_u"]))
    np.testing.assert_array_equal(oracle.bf16_bits_to_f64(r["z"][0]), _row(case["expect_z"]))
    assert int(r["zs"][0, 0]) == case["expect_scale"]
    codes = case["expect_codes"]
    assert np.all(r["zq"][0, 0::2] == int(codes["even"], 16))
    assert np.all(r["zq"][0, 1::2] == int(codes["odd"], 16))


def test_rmsnorm_matches_torch_rms_norm():
    T, S, H = 5, 1, 256
    yb = synth.x_bf16(7, T, H)
    rb = synth.residual_bf16(7, T, S, H)
    gb = synth.norm_weight_bf16(7, H)
    eps = 1e-6
    r = fused.residual_norm_mxfp8(yb, rb, gb, eps)
    u = torch.from_numpy(r["u"].astype(np.float64))
    g = torch.from_numpy(oracle.bf16_bits_to_f64(gb))
    ref = torch.nn.functional.rms_norm(u, (H,), weight=g, eps=float(np.float32(eps))).numpy().astype(np.float32)
    # rsqrt against a divide by sqrt: at most one binary32 step apart after rounding
    diff = np.abs(ref.view(np.int32).astype(np.int64) - r["z32"].view(np.int32).astype(np.int64))
    assert diff.max() <= 1
    assert np.mean(diff == 0) > 0.99


def test_plain_residual_is_a_bf16_addition():
    T, H = 4, 128
    yb = synth.x_bf16(9, T, H)
    rb = synth.residual_bf16(9, T, 1, H)
    r = fused.residual_norm_mxfp8(yb, rb, synth.norm_weight_bf16(9, H), 1e-6)
    to_t = lambda b: torch.from_numpy(b.astype(np.int16)).view(torch.bfloat16).float()
    ref = (to_t(rb[:, 0]) + to_t(yb)).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    np.testing.assert_array_equal(r["resid"][:, 0], ref)
    # one plain stream: u is the new stream itself
    np.testing.assert_array_equal(r["u"], oracle.bf16_bits_to_f64(r["resid"][:, 0]).astype(np.float32))


def test_four_streams_reduce_to_one():
    T, S, H = 3, 4, 64
    yb = synth.x_bf16(4, T, H)
    rb = synth.residual_bf16(4, T, S, H)
    gb = synth.norm_weight_bf16(4, H)
    res = np.broadcast_to(np.eye(S, dtype=np.float32), (T, S, S)).copy()
    post = np.zeros((T, S), np.float32)
    post[:, 2] = 1.0
    pre = np.zeros((T, S), np.float32)
    pre[:, 2] = 1.0
    four = fused.residual_norm_mxfp8(yb, rb, gb, 1e-5, res, post, pre)
    one = fused.residual_norm_mxfp8(yb, rb[:, 2:3], gb, 1e-5)
    for s in (0, 1, 3):
        np.testing.assert_array_equal(four["resid"][:, s], rb[:, s])   # untouched streams
    np.testing.assert_array_equal(four["resid"][:, 2], one["resid"][:, 0])
    for key in ("u", "z", "zq", "zs"):
        np.testing.assert_array_equal(four[key], one[key])


def test_rmsnorm_scale_invariance_with_zero_eps():
    T, H = 3, 96
    yb = synth.x_bf16(8, T, H)
    rb = synth.residual_bf16(8, T, 1, H)
    gb = synth.norm_weight_bf16(8, H)
    twice = lambda b: bits_of(2.0 * oracle.bf16_bits_to_f64(b))
    a = fused.residual_norm_mxfp8(yb, rb, gb, 0.0)
    b = fused.residual_norm_mxfp8(twice(yb), twice(rb), gb, 0.0)
    np.testing.assert_array_equal(b["resid"], twice(a["resid"]))
    np.testing.assert_array_equal(a["z"], b["z"])
    np.testing.assert_array_equal(a["zq"], b["zq"])


def test_epilogue_shape_check():
    with pytest.raises(ValueError):
        fused.residual_norm_mxfp8(np.zeros((2, 32), np.uint16), np.zeros((2, 1, 64), np.uint16),
                                  np.zeros(64, np.uint16), 1e-6)
