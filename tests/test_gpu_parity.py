"""GPU parity: the CUDA path (through the C ABI) against the oracle, on seeded inputs.

Small cases are compared element by element. They span several tiles, ragged
tail tiles, multi-tile experts, k = 1, k = E and a shared expert.
* Routing, placement and x quantisation: bit-exact.
* h quantisation: bit-exact on the GPU's own bf16 h.
* y: within the stated tolerance.
Properties are also checked: determinism, token-permutation invariance, the
empty step, argument errors, and a host-injected bounded-wait timeout.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from moe_expert_layer_top_gb300 import abi, synthetic
from moe_expert_layer_top_gb300.layer import MoEStep, quantize_mxfp4, quantize_mxfp8

from gpu_cases import (CudaStep, bf16_dev_to_bits, check_h_close, check_h_quantizer_bit_exact,
                       check_routing_bit_exact, check_xquant_bit_exact, check_y, oracle_abs_sums, oracle_experts,
                       rel_fro, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import moe_expert_layer_top_gb300 as pkg
    pkg.build.build()
    abi.load()
    assert torch.cuda.is_available()


# ----------------------------------------------------------------- generator and quantiser

def test_device_generator_matches_host_generator():
    import synth.gpu
    n, start = 1 << 20, 12345
    out = torch.empty(n, dtype=torch.int16, device="cuda")
    synth.gpu.normal_bf16(42, synth.stream_gate(7), start, n, synth.expert_sigma(4096), out.data_ptr(),
                          torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    ref = synth.normal_bf16(42, synth.stream_gate(7), start, n, synth.expert_sigma(4096))
    np.testing.assert_array_equal(to_np(out).view(np.uint16), ref)


def _quant_both(bits: np.ndarray):
    x = torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    q, s = quantize_mxfp8(x)
    torch.cuda.synchronize()
    qr, sr = oracle.mxfp8_quantize(oracle.bf16_bits_to_f64(bits))
    np.testing.assert_array_equal(to_np(q), qr)
    np.testing.assert_array_equal(to_np(s), sr)


def test_quantiser_exhaustive_bf16_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_bits_to_f64(bits)
    finite = bits[np.isfinite(vals)]
    pad = (-len(finite)) % 32
    finite = np.concatenate([finite, np.zeros(pad, dtype=np.uint16)])
    _quant_both(finite.reshape(-1, 32))                                   # sorted: similar magnitudes
    rng = np.random.default_rng(0)
    _quant_both(rng.permutation(finite).reshape(-1, 32))                   # mixed magnitudes
    # every pattern against fixed group maxima 1.0, 2^-100 and 2^100 (small values relative to the scale)
    for amax_bits in (0x3F80, 0x0D80, 0x7180):
        g = finite.reshape(-1, 32).copy()
        g[:, 0] = amax_bits
        keep = np.abs(oracle.bf16_bits_to_f64(g)).max(axis=1) <= oracle.bf16_bits_to_f64(np.uint16(amax_bits))
        _quant_both(g[keep])


def _quant4_both(bits: np.ndarray):
    x = torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    q, s = quantize_mxfp4(x)
    torch.cuda.synchronize()
    qr, sr = oracle.mxfp4_quantize(oracle.bf16_bits_to_f64(bits))
    np.testing.assert_array_equal(to_np(s), sr)
    np.testing.assert_array_equal(to_np(q), qr)


def test_mxfp4_quantiser_exhaustive_bf16_patterns():
    """The device MXFP4 quantiser (E2M1 through the hardware conversion) equals
    the oracle's for every finite bf16 pattern, at several group maxima."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_bits_to_f64(bits)
    finite = bits[np.isfinite(vals)]
    pad = (-len(finite)) % 32
    finite = np.concatenate([finite, np.zeros(pad, dtype=np.uint16)])
    _quant4_both(finite.reshape(-1, 32))
    rng = np.random.default_rng(1)
    _quant4_both(rng.permutation(finite).reshape(-1, 32))
    for amax_bits in (0x3F80, 0x0D80, 0x7180, 0x40C0):   # 1.0, 2^-100, 2^100, 6.0
        g = finite.reshape(-1, 32).copy()
        g[:, 0] = amax_bits
        keep = np.abs(oracle.bf16_bits_to_f64(g)).max(axis=1) <= oracle.bf16_bits_to_f64(np.uint16(amax_bits))
        _quant4_both(g[keep])


def test_quantiser_special_groups():
    rows = []
    rows.append(np.zeros(32, dtype=np.uint16))                                 # all +0
    rows.append(np.full(32, 0x8000, dtype=np.uint16))                          # all -0
    rows.append(np.arange(1, 33, dtype=np.uint16))                             # bf16 subnormals only
    rows.append(np.full(32, 0x7F7F, dtype=np.uint16))                          # largest finite bf16
    rows.append(np.array([0x3F80] + [0x3780] * 31, dtype=np.uint16))          # 1.0 with 2^-16 entries
    _quant_both(np.stack(rows))


# ----------------------------------------------------------------- small cases, full comparison

SMALL = [
    # T, H, E, k, I, routing, shared
    (6, 512, 8, 2, 256, "uniform", 0),        # the tiny workload
    (40, 512, 8, 2, 256, "zipf", 0),          # multi-tile experts with ragged tails
    (1, 512, 8, 1, 256, "uniform", 0),        # single row, k = 1
    (13, 512, 8, 8, 256, "uniform", 0),       # k = E: every expert active
    (24, 512, 16, 4, 256, "zipf", 1),         # shared expert
    (20, 1024, 16, 4, 512, "uniform", 0),     # second compiled shape
    (70, 512, 8, 3, 256, "zipf", 1),          # > 64 rows: several bitmap words, hot expert with 9 tiles
    (300, 512, 8, 2, 256, "zipf", 1),         # experts with > 128 rows: several MMA chunks each
]

# Both expert kernels, pinned by flag: the CUDA-core GEMV kernel and the
# tensor-core (block-scaled MXFP8 MMA) kernel.
PATHS = {"gemv": abi.MOE_FLAG_PATH_GEMV, "mma": abi.MOE_FLAG_PATH_MMA}


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("case", SMALL, ids=[f"T{c[0]}_H{c[1]}_E{c[2]}_k{c[3]}_sh{c[6]}" for c in SMALL])
def test_small_case_parity(case, path):
    T, H, E, k, I, routing, shared = case
    g = CudaStep(T, H, E, k, I, routing, shared, seed=42 + T, flags=PATHS[path]).run()
    assert g.status_code == abi.MOE_OK, (abi.moe_status_string(g.status_code), g.diag)
    get = oracle_experts(42 + T, E, H, I)
    sh = oracle.expert_weights_from_synth(42 + T, "shared", H, I) if shared else None
    r = oracle.moe_step(g.x_bits, g.lg, k, get, shared=sh)
    check_routing_bit_exact(g, r)
    check_xquant_bit_exact(g, r)
    check_h_quantizer_bit_exact(g)
    P = T * k + T * shared
    sg, su = oracle_abs_sums(r, T, k, get, sh)
    check_h_close(g, r, np.arange(P), sg, su)
    assert rel_fro(g.t["o"], r["o"]) <= 1e-2
    check_y(g.y_bits, r["y"])
    g.close()


# Tensor-core kernel only: more than 128 rows, where a unit covers two 128-row
# weight blocks with 96-row chunks (H a multiple of 256), or one block with
# 64-row chunks (H = 640); I = 384 gives three gate/up units per chunk.
WIDE = [
    # T, H, E, k, I, routing, shared, weights
    (200, 512, 8, 2, 384, "zipf", 1, "mxfp8"),
    (129, 768, 16, 4, 256, "zipf", 0, "mxfp8"),
    (150, 640, 8, 2, 256, "zipf", 0, "mxfp8"),
    (200, 512, 8, 2, 384, "zipf", 1, "mxfp4"),
]


@pytest.mark.parametrize("case", WIDE, ids=[f"T{c[0]}_H{c[1]}_I{c[4]}_sh{c[6]}_{c[7]}" for c in WIDE])
def test_wide_unit_parity(case):
    T, H, E, k, I, routing, shared, fmt = case
    g = CudaStep(T, H, E, k, I, routing, shared, seed=50 + T, flags=abi.MOE_FLAG_PATH_MMA, fmt=fmt).run()
    assert g.status_code == abi.MOE_OK, (abi.moe_status_string(g.status_code), g.diag)
    get = oracle_experts(50 + T, E, H, I, fmt=fmt)
    sh = oracle.expert_weights_from_synth(50 + T, "shared", H, I, fmt=fmt) if shared else None
    r = oracle.moe_step(g.x_bits, g.lg, k, get, shared=sh)
    check_routing_bit_exact(g, r)
    check_xquant_bit_exact(g, r)
    check_h_quantizer_bit_exact(g)
    sg, su = oracle_abs_sums(r, T, k, get, sh)
    check_h_close(g, r, np.arange(T * k + T * shared), sg, su)
    assert rel_fro(g.t["o"], r["o"]) <= 1e-2
    check_y(g.y_bits, r["y"])
    g.close()


SMALL4 = [
    # T, H, E, k, I, routing, shared, swiglu_limit
    (6, 512, 8, 2, 256, "uniform", 0, 0.0),
    (40, 512, 8, 2, 384, "zipf", 0, 0.0),     # I not a power of two (a multiple of 128)
    (70, 512, 8, 3, 256, "zipf", 1, 0.5),     # shared expert, clipped SwiGLU
    (24, 1024, 16, 4, 640, "uniform", 0, 0.375),
]


@pytest.mark.parametrize("case", SMALL4, ids=[f"T{c[0]}_H{c[1]}_I{c[4]}_sh{c[6]}_lim{c[7]}" for c in SMALL4])
def test_mxfp4_weights_parity(case):
    """MXFP4 expert weights on the tensor-core kernel, against the oracle."""
    T, H, E, k, I, routing, shared, lim = case
    g = CudaStep(T, H, E, k, I, routing, shared, seed=60 + T, fmt="mxfp4", swiglu_limit=lim).run()
    assert g.status_code == abi.MOE_OK, (abi.moe_status_string(g.status_code), g.diag)
    get = oracle_experts(60 + T, E, H, I, fmt="mxfp4")
    sh = oracle.expert_weights_from_synth(60 + T, "shared", H, I, fmt="mxfp4") if shared else None
    r = oracle.moe_step(g.x_bits, g.lg, k, get, shared=sh, swiglu_limit=lim)
    check_routing_bit_exact(g, r)
    check_xquant_bit_exact(g, r)
    check_h_quantizer_bit_exact(g)
    P = T * k + T * shared
    sg, su = oracle_abs_sums(r, T, k, get, sh)
    check_h_close(g, r, np.arange(P), sg, su, lim)
    assert rel_fro(g.t["o"], r["o"]) <= 1e-2
    check_y(g.y_bits, r["y"])
    # the device-prepared MXFP4 weights are the oracle's, bit for bit
    ref = get(0)
    np.testing.assert_array_equal(to_np(g.weights.w_gate[0]), ref.w_gate)
    np.testing.assert_array_equal(to_np(g.weights.s_down[0]), ref.s_down)
    g.close()


@pytest.mark.parametrize("path", list(PATHS))
def test_clipped_swiglu_parity(path):
    T, H, E, k, I, lim = 24, 512, 8, 2, 256, 0.375
    g = CudaStep(T, H, E, k, I, "zipf", 1, seed=71, flags=PATHS[path], swiglu_limit=lim).run()
    assert g.status_code == abi.MOE_OK
    get = oracle_experts(71, E, H, I)
    sh = oracle.expert_weights_from_synth(71, "shared", H, I)
    r = oracle.moe_step(g.x_bits, g.lg, k, get, shared=sh, swiglu_limit=lim)
    r0 = oracle.moe_step(g.x_bits, g.lg, k, get, shared=sh)
    assert np.mean(r["h"] != r0["h"]) > 0.1          # the clip changes h
    check_h_quantizer_bit_exact(g)
    sg, su = oracle_abs_sums(r, T, k, get, sh)
    check_h_close(g, r, np.arange(T * k + T), sg, su, lim)
    check_y(g.y_bits, r["y"])
    g.close()


def test_weights_prepared_on_device_match_oracle_quantisation():
    w = synthetic.make_weights(7, 3, 512, 256, 1)
    for e in range(3):
        ref = oracle.expert_weights_from_synth(7, e, 512, 256)
        np.testing.assert_array_equal(to_np(w.w_gate[e]), ref.w_gate)
        np.testing.assert_array_equal(to_np(w.s_up[e]), ref.s_up)
        np.testing.assert_array_equal(to_np(w.w_down[e]), ref.w_down)
        np.testing.assert_array_equal(to_np(w.s_down[e]), ref.s_down)
    ref = oracle.expert_weights_from_synth(7, "shared", 512, 256)
    np.testing.assert_array_equal(to_np(w.sh_w_up), ref.w_up)


def test_routing_tie_break_on_device():
    T, H, E, k, I = 4, 512, 8, 3, 256
    lg = np.zeros((T, E), dtype=np.float32)
    lg[0] = [1, 2, 2, 2, 0, 0, 0, 0]          # tie among 1, 2, 3
    lg[1] = [0.5] * 8                          # all equal
    lg[2] = [-1, 3, 3, -2, 3, 0, 1, 1]
    lg[3] = np.arange(8)[::-1]
    x = synth.x_bf16(3, T, H)
    g = CudaStep(T, H, E, k, I, x_lg=(x, lg)).run()
    r = oracle.moe_step(x, lg, k, oracle_experts(42, E, H, I))
    check_routing_bit_exact(g, r)
    np.testing.assert_array_equal(g.t["topk_ids"][0], [1, 2, 3])
    check_y(g.y_bits, r["y"])
    g.close()


# ----------------------------------------------------------------- properties

@pytest.mark.parametrize("path", list(PATHS))
def test_deterministic_and_token_permutation_invariant(path):
    T, H, E, k, I = 40, 512, 8, 2, 256
    g = CudaStep(T, H, E, k, I, "zipf", flags=PATHS[path]).run()
    y1 = g.y_bits.copy()
    g.run()
    np.testing.assert_array_equal(g.y_bits, y1)             # same input twice -> same bits
    perm = np.random.default_rng(5).permutation(T)
    g2 = CudaStep(T, H, E, k, I, weights=g.weights, x_lg=(g.x_bits[perm], g.lg[perm]), flags=PATHS[path]).run()
    # each row's arithmetic does not depend on its tile-mates
    np.testing.assert_array_equal(g2.y_bits, y1[perm])
    g.close()
    g2.close()


def test_empty_step_and_argument_errors():
    T, H, E, k, I = 6, 512, 8, 2, 256
    g = CudaStep(T, H, E, k, I)
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.current_stream()
    assert abi.moe_forward(g.step.plan, g.x_dev, g.lg_dev, 0, y, None, None, st) == abi.MOE_OK
    assert abi.moe_forward(g.step.plan, g.x_dev, g.lg_dev, T + 1, y, None, None, st) == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_forward(g.step.plan, g.x_dev, g.lg_dev, -1, y, None, None, st) == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_forward(g.step.plan, g.x_dev.data_ptr() + 2, g.lg_dev, T, y, None, None, st) == \
        abi.MOE_ERR_INVALID_ARG
    g.run()
    assert g.status_code == abi.MOE_OK, (abi.moe_status_string(g.status_code), g.diag)
    g.close()


@pytest.mark.parametrize("path", list(PATHS))
def test_fewer_rows_than_planned(path):
    T, H, E, k, I = 9, 512, 8, 2, 256
    g = CudaStep(T, H, E, k, I, max_rows=64, flags=PATHS[path]).run()
    r = oracle.moe_step(g.x_bits, g.lg, k, oracle_experts(42, E, H, I))
    check_routing_bit_exact(g, r)
    check_y(g.y_bits, r["y"])
    g.close()


@pytest.mark.parametrize("path", list(PATHS))
def test_bounded_wait_timeout_is_reported_and_recoverable(path):
    """Host-injected fault: one tile (chunk) never publishes its ready count. The
    down units' bounded wait gives up, the step reports MOE_ERR_TIMEOUT, and the
    GPU stays usable: a normal plan afterwards matches the oracle."""
    T, H, E, k, I = 6, 512, 8, 2, 256
    g = CudaStep(T, H, E, k, I, flags=abi.MOE_FLAG_TEST_SKIP_READY | PATHS[path], timeout_ns=20_000_000).run()
    assert g.status_code == abi.MOE_ERR_TIMEOUT
    g.close()
    ok = CudaStep(T, H, E, k, I).run()
    assert ok.status_code == abi.MOE_OK
    r = oracle.moe_step(ok.x_bits, ok.lg, k, oracle_experts(42, E, H, I))
    check_y(ok.y_bits, r["y"])
    ok.close()


def test_forward_host_matches_device_forward():
    """Pinned buffers: the kernels read x and the logits and write y in host memory."""
    T, H, E, k, I = 6, 512, 8, 2, 256
    g = CudaStep(T, H, E, k, I).run()
    xh = torch.from_numpy(g.x_bits.view(np.int16).copy()).pin_memory()
    lh = torch.from_numpy(g.lg.copy()).pin_memory()
    yh = torch.empty((T, H), dtype=torch.int16).pin_memory()
    assert g.step.forward_host(xh, lh, yh) == abi.MOE_OK
    np.testing.assert_array_equal(yh.numpy().view(np.uint16), g.y_bits)
    g.close()


@pytest.mark.parametrize("pinned", ["none", "x", "y"])
def test_forward_host_pageable_buffers(pinned):
    """Pageable buffers take copies through the plan's device buffers, alone or
    mixed with pinned ones; the result is the same as the device-side step."""
    T, H, E, k, I = 6, 512, 8, 2, 256
    g = CudaStep(T, H, E, k, I).run()
    xh = torch.from_numpy(g.x_bits.view(np.int16).copy())
    lh = torch.from_numpy(g.lg.copy())
    yh = torch.full((T, H), -1, dtype=torch.int16)
    if pinned == "x":
        xh = xh.pin_memory()
    if pinned == "y":
        yh = yh.pin_memory()
    assert g.step.forward_host(xh, lh, yh) == abi.MOE_OK
    np.testing.assert_array_equal(yh.numpy().view(np.uint16), g.y_bits)
    g.close()


def test_path_flags_are_exclusive():
    T, H, E, k, I = 6, 512, 8, 2, 256
    w = synthetic.make_weights(1, E, H, I, 0, torch.device("cuda", 0))
    with pytest.raises(abi.MoeError):
        MoEStep(H, I, E, k, w, T, 0, abi.MOE_FLAG_PATH_GEMV | abi.MOE_FLAG_PATH_MMA)


def test_default_path_is_the_tensor_core_kernel():
    """Without a path flag every step runs the MMA kernel: its output is the
    pinned MMA kernel's, bit for bit, and matches the oracle."""
    H, E, k, I = 512, 8, 2, 256
    for T in (6, 40):
        g = CudaStep(T, H, E, k, I, "zipf", seed=5).run()
        assert g.status_code == abi.MOE_OK
        pinned = CudaStep(T, H, E, k, I, "zipf", seed=5, weights=g.weights, flags=abi.MOE_FLAG_PATH_MMA).run()
        np.testing.assert_array_equal(g.y_bits, pinned.y_bits)
        r = oracle.moe_step(g.x_bits, g.lg, k, oracle_experts(5, E, H, I))
        check_y(g.y_bits, r["y"])
        g.close()
        pinned.close()


def test_timing_flag_records_expert_kernel():
    T, H, E, k, I = 6, 512, 8, 2, 256
    g = CudaStep(T, H, E, k, I, flags=abi.MOE_FLAG_TIMING)
    for _ in range(3):
        g.run()
    ms, n = g.step.kernel_times()
    assert n == 3 and ms > 0
    g.close()


@pytest.mark.parametrize("path,fused", [("mma", False), ("gemv", False), ("mma", True)])
def test_back_to_back_steps_match_isolated_steps(path, fused):
    """Consecutive steps on one plan, enqueued with no synchronisation between
    them, overlap through programmatic dependent launch (the route kernel of a
    step starts while the previous step's last kernel finishes). Alternating
    between two inputs, every step's y must equal that input's isolated step
    bit for bit: the route kernel must not reset the plan's counters or lists
    while the previous expert kernel still reads them."""
    H, E, k, I, T = 512, 16, 4, 256, 40
    w = synthetic.make_weights(31, E, H, I, 1)
    step = MoEStep(H, I, E, k, w, T, 1, PATHS[path])
    ins = [synthetic.make_inputs(31 + i, T, H, E, k, "zipf") for i in range(2)]
    resid = torch.from_numpy(synth.residual_bf16(5, T, 1, H).view(np.int16).copy()).view(torch.bfloat16).cuda()
    gamma = torch.from_numpy(synth.norm_weight_bf16(5, H).view(np.int16).copy()).view(torch.bfloat16).cuda()

    def one(i):
        x, lg = ins[i][0], ins[i][1]
        if fused:
            return step.forward_fused(x, logits=lg, resid=resid, norm_weight=gamma)["zq"]
        return step.forward(x, lg)
    ref = []
    for i in range(2):
        ref.append(one(i).clone())
        torch.cuda.synchronize()
    outs = [one(n % 2) for n in range(12)]          # back to back, no sync
    torch.cuda.synchronize()
    assert step.status() == abi.MOE_OK
    for n, y in enumerate(outs):
        assert torch.equal(y, ref[n % 2]), n
    step.close()
