"""The h check of the GPU parity tests, on the CPU: a device-like computation
(binary32 sums in another order, binary32 SiLU) stays inside the envelope, and
planted mistakes (one 32-group's scale off by a factor of two, gate and up
swapped) fall outside it. The mistakes are planted in a copy of the oracle's
arithmetic here; no GPU is involved."""
import numpy as np

import oracle
import synth
from gpu_cases import h_envelope

T, H, I = 12, 512, 256
SEED = 5


def _setup():
    w = oracle.expert_weights_from_synth(SEED, 3, H, I)
    x_bits = synth.x_bf16(SEED, T, H)
    xq, xs = oracle.mxfp8_quantize(oracle.bf16_bits_to_f64(x_bits))
    x = oracle.mxfp8_dequantize(xq, xs)
    return w, xq, xs, x


def _device_like(x, wg, wu):
    """g, u as a device might form them: binary32 partial sums per 32-group,
    groups added in reverse order in binary32, then bf16; h in binary32."""
    def proj(wm):
        acc = np.zeros((x.shape[0], wm.shape[0]), dtype=np.float32)
        for gi in reversed(range(H // 32)):
            sl = slice(32 * gi, 32 * gi + 32)
            part = np.zeros_like(acc)
            for kk in range(sl.start, sl.stop):
                part = (part + np.float32(1) * (x[:, kk:kk + 1] * wm[:, kk][None, :]).astype(np.float32)).astype(
                    np.float32)
            acc = (acc + part).astype(np.float32)
        return oracle.f32_to_bf16_bits(acc)
    gb, ub = proj(wg), proj(wu)
    g32 = oracle.bf16_bits_to_f64(gb).astype(np.float32)
    u32 = oracle.bf16_bits_to_f64(ub).astype(np.float32)
    silu = (g32 / (np.float32(1) + np.exp(-g32))).astype(np.float32)
    return oracle.f32_to_bf16_bits((silu * u32).astype(np.float32))


def _inside(h_bits, g_ref, u_ref, sg, su):
    lo, hi = h_envelope(g_ref, u_ref, sg, su, H)
    v = oracle.bf16_bits_to_f64(h_bits)
    return (v >= lo) & (v <= hi)


def test_device_like_h_inside_envelope():
    w, xq, xs, x = _setup()
    g_ref, u_ref, h_ref, *_ = oracle.expert_mlp(xq, xs, w)
    wg, wu = w.dequant("gate"), w.dequant("up")
    sg, su = np.abs(x) @ np.abs(wg).T, np.abs(x) @ np.abs(wu).T
    h_dev = _device_like(x, wg, wu)
    assert np.all(_inside(h_dev, g_ref, u_ref, sg, su))
    assert np.mean(h_dev != h_ref) < 0.05          # most values agree bit for bit anyway


def test_planted_scale_error_leaves_envelope():
    w, xq, xs, x = _setup()
    g_ref, u_ref, _, *_ = oracle.expert_mlp(xq, xs, w)
    wg, wu = w.dequant("gate"), w.dequant("up")
    sg, su = np.abs(x) @ np.abs(wg).T, np.abs(x) @ np.abs(wu).T
    bad = wg.copy()
    bad[5, 96:128] *= 2.0                            # one 32-group of weight row 5 with its scale code + 1
    h_bad = _device_like(x, bad, wu)
    assert not np.all(_inside(h_bad[:, 5], g_ref[:, 5], u_ref[:, 5], sg[:, 5], su[:, 5]))
    bad_x = x.copy()
    bad_x[2, 32:64] *= 0.5                           # one 32-group of token row 2 with its scale code - 1
    h_bad = _device_like(bad_x, wg, wu)
    assert not np.all(_inside(h_bad[2], g_ref[2], u_ref[2], sg[2], su[2]))


def test_planted_gate_up_swap_leaves_envelope():
    w, xq, xs, x = _setup()
    g_ref, u_ref, _, *_ = oracle.expert_mlp(xq, xs, w)
    wg, wu = w.dequant("gate"), w.dequant("up")
    sg, su = np.abs(x) @ np.abs(wg).T, np.abs(x) @ np.abs(wu).T
    h_bad = _device_like(x, wu, wg)
    assert np.mean(~_inside(h_bad, g_ref, u_ref, sg, su)) > 0.5


def test_binary32_silu_overflow_tail_inside_envelope():
    """g = -90: binary32 exp(90) overflows and g / (1 + exp(-g)) gives -0, so h = 0
    where the exact h is about -7e-38 u. That stays inside the envelope; a
    value of the wrong size there does not."""
    g_bits = oracle.f32_to_bf16_bits(np.array([[-90.0, -100.0, -20.0]], dtype=np.float32))
    u_bits = oracle.f32_to_bf16_bits(np.array([[31.0, -5.0, 3.0]], dtype=np.float32))
    z = np.zeros((1, 3))
    lo, hi = h_envelope(g_bits, u_bits, z, z, H)
    assert lo[0, 0] <= 0.0 <= hi[0, 0] and lo[0, 1] <= 0.0 <= hi[0, 1]
    exact = -20.0 / (1.0 + np.exp(20.0)) * 3.0
    assert not (lo[0, 2] <= 0.0 <= hi[0, 2]) and lo[0, 2] <= exact <= hi[0, 2]


def test_pooled_oracle_equals_the_plain_step():
    """full_oracle (the expert MLPs of several steps in spawned processes, as the
    full-size GPU tests use it) gives exactly what oracle.moe_step gives."""
    from gpu_cases import full_oracle
    T, E, k = 40, 8, 2
    x = synth.x_bf16(5, T, H)
    lg = synth.router_logits(5, T, E, k, "zipf")
    x2 = synth.x_bf16(6, 6, H)
    lg2 = synth.router_logits(6, 6, E, k, "uniform")
    ref, hashes = full_oracle(5, {"a": (x, lg, k, True), "b": (x2, lg2, k, False)}, H, I)
    get = lambda e: oracle.expert_weights_from_synth(5, e, H, I)  # noqa: E731
    sh = oracle.expert_weights_from_synth(5, "shared", H, I)
    r = oracle.moe_step(x, lg, k, get, shared=sh)
    for n in ("ids", "w", "xq", "xs", "g", "u", "h", "hq", "hs", "o", "y"):
        np.testing.assert_array_equal(ref["a"][n], r[n])
    np.testing.assert_array_equal(ref["b"]["y"], oracle.moe_step(x2, lg2, k, get)["y"])
    import oracle_pool
    assert hashes["shared"]["w_up"] == oracle_pool.sha256_of(sh.w_up)
