"""The seeded generator: published SplitMix64 outputs, slicing and moments.

The device implementation of the same counter generator is checked against
this one bit for bit in tests/test_gpu_parity.py.
"""
import numpy as np

import synth


def test_splitmix64_published_sequence():
    # SplitMix64 (Steele, Lea, Flood 2014; Vigna's splitmix64.c) from state 1234567:
    # the first five outputs of next().
    key = np.uint64(1234567)
    idx = np.arange(1, 6, dtype=np.uint64)
    with np.errstate(over="ignore"):
        out = synth._mix64(key + idx * np.uint64(synth.GOLDEN))
    assert [int(v) for v in out] == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                                     4593380528125082431, 16408922859458223821]


def test_counter_slices_agree():
    a = synth.counter_u64(42, 7, 0, 1000)
    b = synth.counter_u64(42, 7, 400, 300)
    np.testing.assert_array_equal(a[400:700], b)
    w = synth.expert_weight_bf16(42, synth.stream_gate(3), 64, 512)
    w2 = synth.expert_weight_bf16(42, synth.stream_gate(3), 64, 512, row_start=10, row_count=5)
    np.testing.assert_array_equal(w[10:15], w2)


def test_normal_moments():
    v = synth.bf16_bits_to_float32(synth.normal_bf16(42, 5, 0, 1 << 20, 0.25)).astype(np.float64)
    assert abs(v.mean()) < 2e-3
    assert abs(v.std() - 0.25) < 2e-3
    assert np.abs(v).max() <= 0.25 * 3.4642 * 1.01


def test_logits_margin_and_zipf_popularity():
    lg = synth.router_logits(42, 96, 256, 8, "zipf")
    s = -np.sort(-lg.astype(np.float64), axis=1)
    assert np.all(s[:, :8] - s[:, 1:9] >= 1e-3)
    ids = np.argsort(-lg, axis=1, kind="stable")[:, :8]
    counts = np.bincount(ids.ravel(), minlength=256)
    assert counts[0] > 40 and counts[0] == counts.max()         # Zipf(1.1): expert 0 is hottest
    lu = synth.router_logits(42, 24, 256, 8, "uniform")
    cu = np.bincount(np.argsort(-lu, axis=1, kind="stable")[:, :8].ravel(), minlength=256)
    assert cu.max() <= 6
