"""Pins for the oracle's expert MLP and whole MoE step.

Each check compares the oracle with something that is not itself:
* The SwiGLU MLP is checked against torch's F.linear and F.silu and its
  dtype casts, with the same rounding points. A swapped gate/up, a missing
  transpose or a wrong activation fails this.
* E = 1, k = 1 reduces to one dense expert MLP with weight exactly 1.
* k = E reduces to a dense softmax mixture over all experts. The weights are
  checked against torch.softmax in fp64.
* The shared expert alone (routed experts all zero) is a dense MLP.
* Permuting tokens permutes y exactly. Relabelling experts leaves y unchanged.
"""
import numpy as np
import torch
import torch.nn.functional as F

import oracle
import synth
from oracle import ExpertWeights


def _bf16_tensor(bits):
    return torch.from_numpy(np.asarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)


def _deq_torch(q, s):
    """Dequantise with torch's own float8_e4m3fn decode and exp2 (a library routine)."""
    qt = torch.from_numpy(np.asarray(q, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64)
    st = torch.exp2(torch.from_numpy(np.asarray(s, dtype=np.int64)).to(torch.float64) - 127.0)
    return (qt.reshape(*qt.shape[:-1], -1, 32) * st[..., None]).reshape(qt.shape)


def _expert(seed, e, H, I):
    return oracle.expert_weights_from_synth(seed, e, H, I)


def test_dequantize_matches_torch_float8():
    w = _expert(1, 0, 512, 256)
    np.testing.assert_array_equal(oracle.mxfp8_dequantize(w.w_gate, w.s_gate),
                                  _deq_torch(w.w_gate, w.s_gate).numpy())


def test_expert_mlp_matches_torch_swiglu():
    H, I = 512, 256
    w = _expert(3, 1, H, I)
    x = synth.x_bf16(3, 5, H)
    xq, xs = oracle.mxfp8_quantize(oracle.bf16_bits_to_f64(x))
    g, u, h, hq, hs, o = oracle.step.expert_mlp(xq, xs, w)
    X = _deq_torch(xq, xs)
    gt = F.linear(X, _deq_torch(w.w_gate, w.s_gate)).to(torch.float32).to(torch.bfloat16)
    ut = F.linear(X, _deq_torch(w.w_up, w.s_up)).to(torch.float32).to(torch.bfloat16)
    ht = (F.silu(gt.to(torch.float64)) * ut.to(torch.float64)).to(torch.float32).to(torch.bfloat16)
    np.testing.assert_array_equal(g, gt.view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(u, ut.view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(h, ht.view(torch.int16).numpy().view(np.uint16))
    # The MXFP8 quantiser is pinned in test_oracle_formats; its output goes through torch's decode here.
    ot = F.linear(_deq_torch(hq, hs), _deq_torch(w.w_down, w.s_down)).to(torch.float32).numpy()
    assert np.all(np.abs(o.astype(np.float64) - ot) <= np.spacing(np.abs(ot)))  # fp64 sum order may differ


def _tiny_inputs(seed, T, H, E, k, I, routing="uniform"):
    x = synth.x_bf16(seed, T, H)
    lg = synth.router_logits(seed, T, E, k, routing)
    ex = {e: _expert(seed, e, H, I) for e in range(E)}
    return x, lg, ex


def test_single_expert_reduces_to_dense_mlp():
    T, H, I = 7, 512, 256
    x, lg, ex = _tiny_inputs(4, T, H, 1, 1, I)
    r = oracle.moe_step(x, lg, 1, ex)
    assert np.all(r["w"] == 1.0)
    xq, xs = oracle.mxfp8_quantize(oracle.bf16_bits_to_f64(x))
    *_, o = oracle.step.expert_mlp(xq, xs, ex[0])
    np.testing.assert_array_equal(r["y"], oracle.f32_to_bf16_bits(o))
    assert r["tiles"][0] == 1 and r["counts"][0] == T


def test_all_experts_reduce_to_dense_softmax_mixture():
    T, H, E, I = 5, 512, 4, 256
    x, lg, ex = _tiny_inputs(6, T, H, E, E, I)
    r = oracle.moe_step(x, lg, E, ex)
    p = torch.softmax(torch.from_numpy(lg.astype(np.float64)), dim=1).numpy()
    xq, xs = oracle.mxfp8_quantize(oracle.bf16_bits_to_f64(x))
    ref = np.zeros((T, H))
    for e in range(E):
        *_, o = oracle.step.expert_mlp(xq, xs, ex[e])
        ref += p[:, e:e + 1] * o.astype(np.float64)
    y = oracle.bf16_bits_to_f64(r["y"])
    # y is one bf16 rounding of a binary32 sum away from the fp64 mixture
    assert np.all(np.abs(y - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6 * np.abs(ref).max())
    # every (row, slot) weight equals the softmax probability of the expert chosen there
    np.testing.assert_allclose(r["w"], np.take_along_axis(p, r["ids"].astype(np.int64), 1), rtol=1e-6)


def test_shared_expert_alone_is_a_dense_mlp():
    T, H, E, k, I = 6, 512, 4, 2, 256
    x, lg, ex = _tiny_inputs(8, T, H, E, k, I)
    zero = ExpertWeights(*(np.zeros_like(a) for a in (ex[0].w_gate, ex[0].s_gate, ex[0].w_up,
                                                      ex[0].s_up, ex[0].w_down, ex[0].s_down)))
    sh = _expert(8, "shared", H, I)
    r = oracle.moe_step(x, lg, k, {e: zero for e in range(E)}, shared=sh)
    xq, xs = oracle.mxfp8_quantize(oracle.bf16_bits_to_f64(x))
    *_, o = oracle.step.expert_mlp(xq, xs, sh)
    np.testing.assert_array_equal(r["y"], oracle.f32_to_bf16_bits(o))


def test_token_permutation_and_expert_relabelling():
    T, H, E, k, I = 12, 512, 8, 2, 256
    x, lg, ex = _tiny_inputs(10, T, H, E, k, I)
    base = oracle.moe_step(x, lg, k, ex)["y"]
    perm = np.random.default_rng(0).permutation(T)
    y_p = oracle.moe_step(x[perm], lg[perm], k, ex)["y"]
    np.testing.assert_array_equal(y_p, base[perm])
    relabel = np.random.default_rng(1).permutation(E)        # new id of old expert e is relabel[e]
    lg_r = np.empty_like(lg)
    lg_r[:, relabel] = lg
    ex_r = {int(relabel[e]): ex[e] for e in range(E)}
    np.testing.assert_array_equal(oracle.moe_step(x, lg_r, k, ex_r)["y"], base)


def test_row_subset_matches_full_step():
    T, H, E, k, I = 10, 512, 8, 2, 256
    x, lg, ex = _tiny_inputs(12, T, H, E, k, I)
    full = oracle.moe_step(x, lg, k, ex)
    part = oracle.moe_step(x, lg, k, ex, rows=[2, 7])
    np.testing.assert_array_equal(part["y"][[2, 7]], full["y"][[2, 7]])
    np.testing.assert_array_equal(part["ids"], full["ids"])


# ----------------------------------------------------------------------------- MXFP4 weights, clipped SwiGLU

def _deq4_torch(q, s):
    """MXFP4 values from the packed codes with torch ops: nibbles split with
    integer ops, the E2M1 value table the OCP MX spec prints, exp2 scales."""
    table = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=torch.float64)
    p = torch.from_numpy(np.asarray(q, dtype=np.uint8).astype(np.int64))
    codes = torch.stack([p & 0xF, p >> 4], dim=-1).reshape(*p.shape[:-1], -1)
    vals = table[codes & 7] * torch.where((codes & 8) != 0, -1.0, 1.0).to(torch.float64)
    st = torch.exp2(torch.from_numpy(np.asarray(s, dtype=np.int64)).to(torch.float64) - 127.0)
    return (vals.reshape(*vals.shape[:-1], -1, 32) * st[..., None]).reshape(vals.shape)


def _torch_swiglu(X, w, deq, limit=0.0):
    gt = F.linear(X, deq(w.w_gate, w.s_gate)).to(torch.float32).to(torch.bfloat16)
    ut = F.linear(X, deq(w.w_up, w.s_up)).to(torch.float32).to(torch.bfloat16)
    g64, u64 = gt.to(torch.float64), ut.to(torch.float64)
    if limit > 0:
        g64 = torch.clamp(g64, max=limit)
        u64 = torch.clamp(u64, min=-limit, max=limit)
    ht = (F.silu(g64) * u64).to(torch.float32).to(torch.bfloat16)
    return gt, ut, ht


def test_mxfp4_dequantize_matches_torch_table_decode():
    w = oracle.expert_weights_from_synth(2, 0, 512, 256, fmt="mxfp4")
    assert w.w_gate.shape == (256, 256) and w.s_gate.shape == (256, 16)
    np.testing.assert_array_equal(w.dequant("gate"), _deq4_torch(w.w_gate, w.s_gate).numpy())
    np.testing.assert_array_equal(w.dequant("down"), _deq4_torch(w.w_down, w.s_down).numpy())


def test_expert_mlp_mxfp4_weights_matches_torch_swiglu():
    H, I = 512, 256
    w = oracle.expert_weights_from_synth(3, 1, H, I, fmt="mxfp4")
    x = synth.x_bf16(3, 5, H)
    xq, xs = oracle.mxfp8_quantize(oracle.bf16_bits_to_f64(x))
    g, u, h, hq, hs, o = oracle.step.expert_mlp(xq, xs, w)
    X = _deq_torch(xq, xs)
    gt, ut, ht = _torch_swiglu(X, w, _deq4_torch)
    np.testing.assert_array_equal(g, gt.view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(u, ut.view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(h, ht.view(torch.int16).numpy().view(np.uint16))
    ot = F.linear(_deq_torch(hq, hs), _deq4_torch(w.w_down, w.s_down)).to(torch.float32).numpy()
    assert np.all(np.abs(o.astype(np.float64) - ot) <= np.spacing(np.abs(ot)))


def test_clipped_swiglu_matches_torch_clamp():
    H, I, limit = 512, 256, 0.375
    w = oracle.expert_weights_from_synth(4, 2, H, I)
    x = synth.x_bf16(4, 7, H)
    xq, xs = oracle.mxfp8_quantize(oracle.bf16_bits_to_f64(x))
    g, u, h, _, _, _ = oracle.step.expert_mlp(xq, xs, w, swiglu_limit=limit)
    gt, ut, ht = _torch_swiglu(_deq_torch(xq, xs), w, _deq_torch, limit)
    np.testing.assert_array_equal(h, ht.view(torch.int16).numpy().view(np.uint16))
    gf, uf = oracle.bf16_bits_to_f64(g), oracle.bf16_bits_to_f64(u)
    assert np.mean(gf > limit) > 0.1 and np.mean(np.abs(uf) > limit) > 0.1  # the clip is active
    _, _, h0, _, _, _ = oracle.step.expert_mlp(xq, xs, w)
    assert np.mean(h != h0) > 0.1


def test_clip_with_a_large_limit_changes_nothing():
    H, I = 512, 256
    w = oracle.expert_weights_from_synth(5, 3, H, I)
    x = synth.x_bf16(5, 4, H)
    xq, xs = oracle.mxfp8_quantize(oracle.bf16_bits_to_f64(x))
    a = oracle.step.expert_mlp(xq, xs, w)
    b = oracle.step.expert_mlp(xq, xs, w, swiglu_limit=1e30)
    for p, q in zip(a, b):
        np.testing.assert_array_equal(p, q)


def test_expert_weights_from_bf16_is_the_synth_path_and_lossless_on_grid_values():
    """expert_weights_from_bf16 on the generator's bits equals
    expert_weights_from_synth; on grid values (synth.exact_case) both formats
    quantise without loss."""
    import synth
    H, I = 256, 128
    a = oracle.expert_weights_from_synth(3, 1, H, I)
    b = oracle.expert_weights_from_bf16(synth.expert_weight_bf16(3, synth.stream_gate(1), I, H),
                                        synth.expert_weight_bf16(3, synth.stream_up(1), I, H),
                                        synth.expert_weight_bf16(3, synth.stream_down(1), H, I))
    for n in ("w_gate", "s_gate", "w_up", "s_up", "w_down", "s_down"):
        np.testing.assert_array_equal(getattr(a, n), getattr(b, n))
    c = synth.exact_case(4, 8, H, 2, 2, I)
    for fmt in ("mxfp8", "mxfp4"):
        w = oracle.expert_weights_from_bf16(c["gate"][1], c["up"][1], c["down"][1], fmt)
        for n in ("gate", "up", "down"):
            np.testing.assert_array_equal(w.dequant(n), oracle.bf16_bits_to_f64(c[n][1]))


def test_exact_case_preconditions_hold():
    """The structured inputs of the exact GPU parity case keep every binary32
    sum of the step exact (the same checks the GPU test makes before it
    compares bit for bit), for both weight formats and every case it runs."""
    import synth
    from test_gpu_exact import EXACT, _exact_sums_hold
    H, E, k, I = 512, 8, 2, 256
    for fmt in ("mxfp8", "mxfp4"):
        for T, routing, shared in EXACT:
            c = synth.exact_case(9, T, H, E, k, I, shared, routing)
            ws = [oracle.expert_weights_from_bf16(c["gate"][e], c["up"][e], c["down"][e], fmt) for e in range(E)]
            sh = oracle.expert_weights_from_bf16(c["sh_gate"], c["sh_up"], c["sh_down"], fmt) if shared else None
            r = oracle.moe_step(c["x"], c["logits"], k, ws.__getitem__, shared=sh)
            _exact_sums_hold(r, ws.__getitem__, sh, T, k)
            assert np.mean([len(set(row)) for row in r["hs"]]) > 2.0   # h's scale codes vary along I
