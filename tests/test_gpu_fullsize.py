"""GPU parity at the full workload sizes (H=4096, E=256, top-8, I=2048), in the
launch configuration the benchmark times.

* Routing, placement and x quantisation are compared in full, bit for bit.
* The h quantiser is compared in full against the oracle's quantisation of
  the GPU's own bf16 h.
* The canonical MXFP8 weights prepared on the device are compared bit for bit
  for the sampled experts.
* y and o are compared on sampled token rows. The oracle computes those rows
  alone, with every expert they touch.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_top_gb300 import abi, synthetic
from moe_expert_layer_top_gb300.layer import MoEWeightsMXFP8

import synth
from gpu_cases import (CudaStep, check_h_close, check_h_quantizer_bit_exact, check_routing_bit_exact,
                       check_xquant_bit_exact, check_y, oracle_experts, rel_fro, to_np)

pytestmark = pytest.mark.gpu

SEED = synth.BASE_SEED
_CACHE = {}


@pytest.fixture(scope="module")
def weights():
    import moe_expert_layer_top_gb300 as pkg
    pkg.build.build()
    w = synthetic.make_weights(SEED, 256, 4096, 2048, shared=1, device=torch.device("cuda", 0))
    torch.cuda.synchronize()
    yield w
    del w
    torch.cuda.empty_cache()


def routed_only(w: MoEWeightsMXFP8) -> MoEWeightsMXFP8:
    return MoEWeightsMXFP8(w.w_gate, w.s_gate, w.w_up, w.s_up, w.w_down, w.s_down)


# flags 0: the expert kernel the benchmark times (the tensor-core kernel); the
# pinned cases run the CUDA-core GEMV kernel on the same workload.
FULL = [("bs1", 0), ("bs4", 0), ("bs16", 0), ("bs64", 0),
        ("bs1", abi.MOE_FLAG_PATH_GEMV), ("bs4", abi.MOE_FLAG_PATH_GEMV), ("bs16", abi.MOE_FLAG_PATH_GEMV)]


@pytest.mark.parametrize("name,flags", FULL, ids=[f"{n}_{'default' if f == 0 else 'mma' if f == abi.MOE_FLAG_PATH_MMA else 'gemv'}"
                                                  for n, f in FULL])
def test_fullsize_parity(name, flags, weights):
    wl = synth.WORKLOADS[name]
    w = weights if wl.shared else routed_only(weights)
    g = CudaStep(wl.T, wl.H, wl.E, wl.k, wl.I, wl.routing, wl.shared, seed=SEED, weights=w, flags=flags).run()
    assert g.status_code == abi.MOE_OK, (abi.moe_status_string(g.status_code), g.diag)
    # sampled rows: the first and the last token row
    rows = [0, wl.T - 1]
    get = oracle_experts(SEED, wl.E, wl.H, wl.I, _CACHE)
    sh = None
    if wl.shared:
        if "shared" not in _CACHE:
            _CACHE["shared"] = oracle.expert_weights_from_synth(SEED, "shared", wl.H, wl.I)
        sh = _CACHE["shared"]
    r = oracle.moe_step(g.x_bits, g.lg, wl.k, get, shared=sh, rows=rows)
    check_routing_bit_exact(g, r)
    check_xquant_bit_exact(g, r)
    check_h_quantizer_bit_exact(g)                       # every pair of the step
    pairs = [t * wl.k + j for t in rows for j in range(wl.k)]
    if wl.shared:
        pairs += [wl.T * wl.k + t for t in rows]
    check_h_close(g, r, pairs)
    assert rel_fro(g.t["o"][pairs], r["o"][pairs]) <= 1e-2
    check_y(g.y_bits[rows], r["y"][rows])
    # the device-prepared MXFP8 weights of the sampled experts, bit for bit
    for e in sorted(set(int(v) for v in r["ids"][rows].ravel()))[:2]:
        ref = get(e)
        np.testing.assert_array_equal(to_np(weights.w_gate[e]), ref.w_gate)
        np.testing.assert_array_equal(to_np(weights.s_gate[e]), ref.s_gate)
        np.testing.assert_array_equal(to_np(weights.w_down[e]), ref.w_down)
        np.testing.assert_array_equal(to_np(weights.s_down[e]), ref.s_down)
    # properties that hold at any size: every pair placed exactly once, tiles <= 8 rows
    slot = g.t["slot"]
    e_of, rank = slot >> 16, slot & 0xFFFF
    assert len(set(zip(e_of.ravel().tolist(), rank.ravel().tolist()))) == wl.T * wl.k
    assert np.all(rank < g.t["counts"][e_of])
    assert np.all(np.abs(g.t["topk_w"].sum(axis=1) - 1.0) <= 1e-6)
    g.close()


@pytest.mark.parametrize("name", ["bs1", "bs64"])
def test_fullsize_mxfp4_intermediate_2304_clipped(name):
    """The pages' checkpoint shape: MXFP4 expert weights, I = 4 x 576 = 2304,
    clipped SwiGLU (limit 1.0 here; the pages give none), on the tensor-core
    kernel at the full expert pool, sampled rows against the oracle."""
    import dataclasses
    wl = dataclasses.replace(synth.WORKLOADS[name], I=2304)
    lim = 1.0
    w = synthetic.make_weights(SEED, wl.E, wl.H, wl.I, wl.shared, torch.device("cuda", 0), "mxfp4")
    torch.cuda.synchronize()
    g = CudaStep(wl.T, wl.H, wl.E, wl.k, wl.I, wl.routing, wl.shared, seed=SEED, weights=w, fmt="mxfp4",
               swiglu_limit=lim).run()
    assert g.status_code == abi.MOE_OK, (abi.moe_status_string(g.status_code), g.diag)
    rows = [0, wl.T - 1]
    get = oracle_experts(SEED, wl.E, wl.H, wl.I, fmt="mxfp4")
    sh = oracle.expert_weights_from_synth(SEED, "shared", wl.H, wl.I, fmt="mxfp4") if wl.shared else None
    r = oracle.moe_step(g.x_bits, g.lg, wl.k, get, shared=sh, rows=rows, swiglu_limit=lim)
    check_routing_bit_exact(g, r)
    check_h_quantizer_bit_exact(g)
    pairs = [t * wl.k + j for t in rows for j in range(wl.k)] + ([wl.T * wl.k + t for t in rows] if wl.shared else [])
    check_h_close(g, r, pairs)
    assert rel_fro(g.t["o"][pairs], r["o"][pairs]) <= 1e-2
    check_y(g.y_bits[rows], r["y"][rows])
    e = int(r["ids"][0, 0])
    np.testing.assert_array_equal(to_np(w.w_down[e]), get(e).w_down)
    g.close()
    del w
    torch.cuda.empty_cache()
