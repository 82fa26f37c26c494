"""Pins for the oracle's number formats (bf16, E4M3, MXFP8).

The oracle is checked against things that are not itself:
* hand-worked examples in tests/golden/mxfp8_examples.json;
* brute-force nearest-value searches over the whole E4M3 grid;
* torch's own float8_e4m3fn and bfloat16 conversions (library routines);
* a second characterisation of the scale rule: the scaled amax lies in [256, 512).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import formats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def all_finite_bf16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_bits_to_f64(bits)
    keep = np.isfinite(vals)
    return bits[keep], vals[keep]


def test_e4m3_table_closed_forms():
    # Values fixed by the E4M3 definition (bias 7, 3 mantissa bits, no infinities).
    d = oracle.e4m3_decode
    assert d(0x7E) == 448.0
    assert d(0x08) == 2.0 ** -6            # smallest normal
    assert d(0x01) == 2.0 ** -9            # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9        # largest subnormal
    assert d(0x38) == 1.0
    assert d(0x78) == 256.0
    assert d(0xFE) == -448.0
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    assert d(0x80) == 0.0 and np.signbit(d(0x80))
    pos = formats.E4M3_TABLE[:0x7F]
    assert np.all(np.diff(pos) > 0)        # codes 0..126 strictly increasing
    assert len(np.unique(pos)) == 127


def test_e4m3_encode_matches_brute_force_on_every_bf16():
    _, v = all_finite_bf16()
    got = oracle.e4m3_encode(v)
    grid_codes = np.array([c for c in range(256) if not np.isnan(formats.E4M3_TABLE[c])])
    grid = formats.E4M3_TABLE[grid_codes]
    a = np.clip(v, -448.0, 448.0)
    dist = np.abs(a[:, None] - grid[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    # several candidates: +0 / -0, or a tie between neighbours -> even mantissa
    exp_codes = np.empty(len(v), dtype=np.int64)
    for i in range(len(v)):
        cs = grid_codes[cand[i]]
        vals = formats.E4M3_TABLE[cs]
        if np.all(vals == 0):
            exp_codes[i] = 0x80 if np.signbit(v[i]) else 0x00
            continue
        # Once the zero pair is resolved, a tie can only be between two
        # neighbours with the same sign.
        cs = cs[(cs & 0x80) == (0x80 if np.signbit(v[i]) else 0)]
        if len(cs) > 1:
            cs = cs[(cs & 1) == 0]
        assert len(cs) == 1
        exp_codes[i] = cs[0]
    np.testing.assert_array_equal(got, exp_codes.astype(np.uint8))


def test_e4m3_encode_matches_torch_in_range():
    _, v = all_finite_bf16()
    v = v[np.abs(v) <= 448.0]
    ref = torch.from_numpy(v).to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(v), ref)


def test_e4m3_roundtrip_and_saturation():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    np.testing.assert_array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes)), codes)
    big = np.array([448.0, 449.0, 463.99, 464.0, 500.0, 1e30, -1e30])
    np.testing.assert_array_equal(oracle.e4m3_encode(big),
                                  np.array([0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE], dtype=np.uint8))


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    f = rng.standard_normal(200000).astype(np.float32) * np.float32(3.0)
    # include exact ties: low half 0x8000 with odd and even kept parts
    ties = (np.arange(1000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    f = np.concatenate([f, ties, np.array([0.0, -0.0, 3.4e38, -3.4e38], dtype=np.float32)])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.f32_to_bf16_bits(f), ref)
    bits, vals = all_finite_bf16()
    ref_vals = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(vals, ref_vals)


def _golden_group(case):
    v = np.full(32, case["filler"], dtype=np.float64)
    for pos, val in case["entries"]:
        v[pos] = val
    return v


def test_mxfp8_hand_worked_examples():
    cases = json.load(open(os.path.join(GOLDEN, "mxfp8_examples.json")))["cases"]
    assert len(cases) >= 8
    for case in cases:
        v = _golden_group(case)
        # every example value is an exact bf16
        assert np.array_equal(oracle.bf16_bits_to_f64(oracle.f32_to_bf16_bits(v.astype(np.float32))), v), case["name"]
        q, s = oracle.mxfp8_quantize(v[None, :])
        assert int(s[0, 0]) == case["expect_scale"], case["name"]
        for key, code in case["expect_codes"].items():
            idx = [i for i in range(32) if i not in [p for p, _ in case["entries"]]] if key == "filler" else [int(key)]
            for i in idx:
                assert int(q[0, i]) == int(code, 16), (case["name"], i)


def test_mxfp8_scale_rule_second_characterisation():
    # Floor rule <=> the scaled amax lies in [256, 512) unless the code is clamped.
    rng = np.random.default_rng(7)
    v = rng.standard_normal((4000, 32)) * np.exp2(rng.integers(-60, 60, size=(4000, 1)))
    v = oracle.bf16_bits_to_f64(oracle.f32_to_bf16_bits(v.astype(np.float32)))
    q, s = oracle.mxfp8_quantize(v)
    amax = np.abs(v).max(axis=1)
    scaled = amax * np.exp2(127.0 - s[:, 0].astype(np.float64))
    assert np.all((scaled >= 256) & (scaled < 512))
    # element error: nearest grid value, i.e. at most half a grid step (or saturation)
    deq = oracle.mxfp8_dequantize(q, s)
    sc = np.exp2(s[:, :1].astype(np.float64) - 127.0)
    x = v / sc
    err = np.abs(deq / sc - np.clip(x, -448, 448))
    step = np.where(np.abs(x) < 2.0 ** -6, 2.0 ** -9, np.exp2(np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -6))) - 3))
    assert np.all(err <= step / 2 + 1e-300)


def test_mxfp8_groups_are_independent_and_along_last_axis():
    rng = np.random.default_rng(3)
    v = oracle.bf16_bits_to_f64(oracle.f32_to_bf16_bits(rng.standard_normal((3, 128)).astype(np.float32)))
    q, s = oracle.mxfp8_quantize(v)
    assert q.shape == (3, 128) and s.shape == (3, 4)
    for g in range(4):
        qg, sg = oracle.mxfp8_quantize(v[:, 32 * g: 32 * g + 32])
        np.testing.assert_array_equal(qg, q[:, 32 * g: 32 * g + 32])
        np.testing.assert_array_equal(sg[:, 0], s[:, g])
    with pytest.raises(ValueError):
        oracle.mxfp8_quantize(np.zeros((1, 48)))


# ----------------------------------------------------------------------------- E2M1 / MXFP4

_G4 = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "mxfp4_examples.json")))


def test_e2m1_decode_matches_the_spec_value_table():
    pos = np.array(_G4["e2m1_positive_values"])
    np.testing.assert_array_equal(oracle.e2m1_decode(np.arange(8)), pos)
    np.testing.assert_array_equal(oracle.e2m1_decode(np.arange(8, 16)), -pos)
    assert np.signbit(oracle.e2m1_decode(8))  # code 0b1000 is -0


def test_e2m1_encode_is_nearest_ties_even_saturating_brute_force():
    grid = oracle.e2m1_decode(np.arange(16))
    rng = np.random.default_rng(4)
    v = np.concatenate([rng.uniform(-8, 8, 20000), np.arange(-80, 81) / 10.0,
                        grid, (grid[:-1] + grid[1:]) / 2.0, [-0.0, 0.0, 1e-9, -1e-9, 100.0, -100.0]])
    got = oracle.e2m1_encode(v)
    for x, c in zip(v, got):
        a = min(abs(x), 6.0)
        d = np.abs(grid[:8] - a)
        best = np.flatnonzero(d == d.min())
        # ties: the even code (mantissa bit 0)
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        if np.signbit(x):
            want |= 8
        assert c == want, (x, c, want)


def test_e2m1_pack_order_and_roundtrip():
    assert oracle.pack_e2m1(np.array([1, 2], dtype=np.uint8))[0] == 0x21  # element 0 in the low nibble
    codes = np.random.default_rng(5).integers(0, 16, size=(3, 64)).astype(np.uint8)
    np.testing.assert_array_equal(oracle.unpack_e2m1(oracle.pack_e2m1(codes)), codes)


def _mx4_group(name):
    g = np.zeros(32)
    if name.startswith("F1"):
        g[:] = 1.0
    elif name.startswith("F2"):
        g[:6] = [6.0, 0.25, 0.75, 2.5, 5.0, 1.25]
    elif name.startswith("F3"):
        g[:2] = [7.5, 1.0]
    elif name.startswith("F4"):
        g[:4] = [-3.0, -0.1, 6.0, -6.0]
    elif name.startswith("F5"):
        g[:2] = [0.046875, 0.0234375]
    return g


@pytest.mark.parametrize("ex", _G4["examples"], ids=[e["name"] for e in _G4["examples"]])
def test_mxfp4_hand_worked_examples(ex):
    q, s = oracle.mxfp4_quantize(_mx4_group(ex["name"])[None, :])
    assert int(s[0, 0]) == ex["scale_code"]
    codes = oracle.unpack_e2m1(q)[0]
    np.testing.assert_array_equal(codes[:len(ex["first_codes"])], ex["first_codes"])
    if "first_bytes" in ex:
        np.testing.assert_array_equal(q[0, :len(ex["first_bytes"])], ex["first_bytes"])


def test_mxfp4_scale_characterisation_and_error_bound():
    rng = np.random.default_rng(6)
    v = rng.standard_normal((64, 128)) * np.exp2(rng.integers(-20, 20, size=(64, 1)))
    q, s = oracle.mxfp4_quantize(v)
    g = v.reshape(64, 4, 32)
    scale = np.exp2(s.astype(np.float64) - 127)
    amax_scaled = np.max(np.abs(g), axis=-1) / scale
    assert np.all((amax_scaled >= 4.0) & (amax_scaled < 8.0))   # 2^(floor(log2 amax) - 2) puts amax in [4, 8)
    deq = oracle.mxfp4_dequantize(q, s).reshape(64, 4, 32)
    a = np.abs(g) / scale[..., None]
    # grid spacing of E2M1 at |x|: 0.5 below 2, 1 in [2, 4), 2 in [4, 6]; above 6 the value saturates to 6
    step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    bound = np.where(a > 6, a - 6, step / 2) * scale[..., None]
    assert np.all(np.abs(deq - g) <= bound + 1e-300)
