"""GPU parity of the steps fused on either side of the MoE step (moe_forward_fused).

In front, the router projection: logits = x . W_r^T (bf16 operands, binary32
sums) in the route kernel.
* The logits are within the binary32 summation bound of the oracle's:
  gamma_d * sum_h |x_h w_h|. Up to 8 rows the kernel sums on CUDA cores (per-lane
  fused multiply-adds, a butterfly, four H quarters): at most H/128 + 8
  roundings per product. Beyond 8 rows it uses tensor-core MMAs (m16n8k16,
  fp32 accumulate) in 16 K slices. d = 40 * H/256 + 64 covers both paths with
  room to spare: up to 17 accumulation steps per MMA, H/256 MMAs in a chain,
  each step allowed two units in the last place (the tensor core may truncate
  rather than round), plus the slice sums.
* Routing, weights and placement are bit-exact against the oracle's top-k
  applied to the GPU's own logits. The decision is taken in the kernel's
  precision.
* The expert ids equal the oracle's from its own logits on every row whose
  top-k margins exceed twice the bound.
Behind, the residual-stream epilogue: one kernel per step, one block per row,
launched right behind the expert kernel.
* New streams are compared with the oracle applied to the GPU's own y:
  bit-exact with one plain stream. With mixing each new value is a binary32
  sum of S + 1 signed terms, so where they cancel its error is bounded by
  the terms' magnitudes, not the result's: every value is within one bf16
  step plus gamma_{S+1} * sum |term| of the oracle's, and at least 99 % are
  equal.
* z is compared with the oracle's z from the GPU's own new streams: within
  one bf16 step plus the binary32 bound of the S-term input combination u
  carried through the normalisation (at least 99 % equal).
* The MXFP8 codes are bit-exact on the GPU's own z.
* The whole chain is within the y tolerance of the oracle's chain.
Source: "Beyond Day-0: Optimizing DeepSeek-V4.1 Flash in SGLang", section 2.1.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from moe_expert_layer_top_gb300 import abi, synthetic
from moe_expert_layer_top_gb300.layer import MoEStep, taps_for

from gpu_cases import bf16_dev_to_bits, check_y, oracle_experts, rel_fro, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import moe_expert_layer_top_gb300 as pkg
    pkg.build.build()
    abi.load()
    assert torch.cuda.is_available()


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16).to(device)


def logits_bound(x_bits, wr_bits) -> np.ndarray:
    """Largest binary32 summation error of a projection logit, per (t, e)."""
    H = x_bits.shape[1]
    d = 40 * max(1, H // 256) + 64
    u = 2.0 ** -24
    gam = d * u / (1 - d * u)
    ax = np.abs(oracle.bf16_bits_to_f64(x_bits))
    aw = np.abs(oracle.bf16_bits_to_f64(wr_bits))
    return gam * (ax @ aw.T) + 1e-30


def topk_margin(lg: np.ndarray, k: int) -> np.ndarray:
    """Smallest gap between adjacent values among each row's k + 1 largest."""
    s = -np.sort(-lg.astype(np.float64), axis=1)[:, : k + 1]
    return np.min(s[:, :-1] - s[:, 1:], axis=1)


def _gamma(n: int) -> float:
    u = 2.0 ** -24
    return n * u / (1 - n * u)


def _bf16_step(v: np.ndarray) -> np.ndarray:
    """One bf16 step at |v| (the normal-range step for 0 and subnormals)."""
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 7)


def check_mixed_epilogue(out, y_gpu, resid, gamma, eps, res, post, pre):
    """New streams and z of a mixed-stream epilogue against the oracle, within
    the binary32 summation bounds (see the module docstring)."""
    T, H = y_gpu.shape
    S = resid.shape[1]
    ref = oracle.residual_norm_mxfp8(y_gpu, resid, gamma, eps, res, post, pre)
    got = oracle.bf16_bits_to_f64(bf16_dev_to_bits(out["resid"]).reshape(T, S, H))
    exp = oracle.bf16_bits_to_f64(ref["resid"])
    r = oracle.bf16_bits_to_f64(resid)
    y = oracle.bf16_bits_to_f64(y_gpu)
    res64, post64, pre64 = (np.asarray(c, dtype=np.float64) for c in (res, post, pre))
    terms = np.einsum("tab,tbh->tah", np.abs(res64), np.abs(r)) + np.abs(post64)[:, :, None] * np.abs(y)[:, None, :]
    lim = np.maximum(_bf16_step(got), _bf16_step(exp)) + _gamma(S + 1) * terms
    assert np.all(np.abs(got - exp) <= lim), np.max(np.abs(got - exp) / lim)
    assert np.mean(got == exp) > 0.99
    # z from the GPU's own new streams
    ref_g = oracle.residual_norm_mxfp8(y_gpu, bf16_dev_to_bits(out["resid"]).reshape(T, S, H), gamma, eps,
                                       np.eye(S, dtype=np.float32)[None].repeat(T, 0), np.zeros((T, S), np.float32),
                                       pre)
    u = np.einsum("ts,tsh->th", pre64, got)
    rms = np.sqrt(np.mean(u * u, axis=1) + float(np.float32(eps)))
    g = np.abs(oracle.bf16_bits_to_f64(gamma))
    z_gpu = oracle.bf16_bits_to_f64(bf16_dev_to_bits(out["z"]))
    z_ref = oracle.bf16_bits_to_f64(ref_g["z"])
    u_err = _gamma(S) * np.einsum("ts,tsh->th", np.abs(pre64), np.abs(got))
    z_lim = np.maximum(_bf16_step(z_gpu), _bf16_step(z_ref)) + g[None, :] * u_err / rms[:, None] \
        + np.abs(z_ref) * 2.0 ** -20
    assert np.all(np.abs(z_gpu - z_ref) <= z_lim), np.max(np.abs(z_gpu - z_ref) / z_lim)
    assert np.mean(z_gpu == z_ref) > 0.99
    return ref


def check_routing_from_gpu_logits(t: dict, lg_gpu: np.ndarray, k: int, E: int):
    ids = oracle.topk_ids(lg_gpu, k)
    w = oracle.softmax_topk_weights(lg_gpu, ids)
    plc = oracle.placement(ids, E)
    np.testing.assert_array_equal(t["topk_ids"], ids)
    np.testing.assert_array_equal(t["topk_w"].view(np.uint32), w.view(np.uint32))
    np.testing.assert_array_equal(t["bitmap"].view(np.uint32), plc["bitmap"])
    np.testing.assert_array_equal(t["counts"], plc["counts"])
    ref_slot = (plc["slot_e"].astype(np.int64) << 16) | (plc["slot_tile"] * 8 + plc["slot_row"])
    np.testing.assert_array_equal(t["slot"].astype(np.int64), ref_slot)
    return ids


# T spans one and two row groups of 32 with a ragged tail; E = 12 leaves a
# partial block of 8 experts.
@pytest.mark.parametrize("T,H,E,k,I,shared", [
    (6, 512, 8, 2, 256, 0),
    (40, 512, 12, 3, 256, 1),
    (70, 1024, 64, 8, 256, 0),
])
def test_router_projection(T, H, E, k, I, shared):
    dev = torch.device("cuda", 0)
    seed = 31
    w = synthetic.make_weights(seed, E, H, I, shared, dev)
    x_bits = synth.x_bf16(seed, T, H)
    wr_bits = synth.router_weight_bf16(seed, E, H)
    step = MoEStep(H, I, E, k, w, T, shared)
    taps, tt = taps_for(T, k, E, H, I, shared, dev)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    out = step.forward_fused(dev_bf16(x_bits), w_router=dev_bf16(wr_bits), taps=taps, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == abi.MOE_OK
    lg_gpu = to_np(out["logits"])
    lg_ref = oracle.router_logits(x_bits, wr_bits)
    bound = logits_bound(x_bits, wr_bits)
    err = np.abs(lg_gpu.astype(np.float64) - lg_ref.astype(np.float64))
    assert np.all(err <= bound + np.abs(lg_ref) * 2.0 ** -24), float(np.max(err / bound))
    t = {n: to_np(v) for n, v in tt.items()}
    ids = check_routing_from_gpu_logits(t, lg_gpu, k, E)
    # rows with clear margins route as the oracle's own logits do
    clear = topk_margin(lg_ref, k) > 2 * np.max(bound, axis=1)
    assert np.mean(clear) > 0.5
    np.testing.assert_array_equal(ids[clear], oracle.topk_ids(lg_ref, k)[clear])
    # the step itself, on the GPU's logits
    get = oracle_experts(seed, E, H, I)
    sh = oracle.expert_weights_from_synth(seed, "shared", H, I) if shared else None
    r = oracle.moe_step(x_bits, lg_gpu, k, get, shared=sh)
    np.testing.assert_array_equal(t["xq"], r["xq"])
    np.testing.assert_array_equal(t["xs"], r["xs"])
    check_y(bf16_dev_to_bits(out["y"]), r["y"])
    # deterministic: a second run gives the same logits and y
    out2 = step.forward_fused(dev_bf16(x_bits), w_router=dev_bf16(wr_bits))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(out2["logits"]).view(np.uint32), lg_gpu.view(np.uint32))
    np.testing.assert_array_equal(bf16_dev_to_bits(out2["y"]), bf16_dev_to_bits(out["y"]))
    step.close()


def test_fused_without_extras_equals_moe_forward():
    dev = torch.device("cuda", 0)
    T, H, E, k, I = 24, 512, 16, 4, 256
    w = synthetic.make_weights(5, E, H, I, 0, dev)
    x, lg, _, _ = synthetic.make_inputs(5, T, H, E, k, "zipf", dev)
    step = MoEStep(H, I, E, k, w, T, 0)
    y0 = step.forward(x, lg)
    out = step.forward_fused(x, logits=lg)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bf16_dev_to_bits(out["y"]), bf16_dev_to_bits(y0))
    step.close()


def _epilogue_inputs(seed, T, S, H, mixed):
    resid = synth.residual_bf16(seed, T, S, H)
    gamma = synth.norm_weight_bf16(seed, H)
    coef = synth.mix_coefficients(seed, T, S) if mixed else (None, None, None)
    return resid, gamma, coef


@pytest.mark.parametrize("T,H,E,k,I,S,mixed,in_place", [
    (6, 512, 8, 2, 256, 1, False, False),
    (37, 1024, 16, 4, 256, 1, False, True),
    (20, 512, 8, 2, 384, 4, True, False),
    (9, 1024, 16, 3, 256, 2, True, True),
    (3, 16384, 4, 2, 128, 2, True, False),   # 512 groups per row: two per thread
])
def test_residual_norm_epilogue(T, H, E, k, I, S, mixed, in_place):
    dev = torch.device("cuda", 0)
    seed = 23
    w = synthetic.make_weights(seed, E, H, I, 0, dev)
    x, lg, x_bits, lg_np = synthetic.make_inputs(seed, T, H, E, k, "uniform", dev)
    resid, gamma, (res, post, pre) = _epilogue_inputs(seed, T, S, H, mixed)
    to_dev = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    eps = 1e-6
    step = MoEStep(H, I, E, k, w, T, 0)
    resid_dev = dev_bf16(resid)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    out = step.forward_fused(x, logits=lg, resid=resid_dev, norm_weight=dev_bf16(gamma), rms_eps=eps,
                             mix_res=to_dev(res), mix_post=to_dev(post), mix_pre=to_dev(pre), in_place=in_place,
                             z_tap=True, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == abi.MOE_OK
    if in_place:
        assert out["resid"].data_ptr() == resid_dev.data_ptr()
    y_gpu = bf16_dev_to_bits(out["y"])
    ref = oracle.residual_norm_mxfp8(y_gpu, resid, gamma, eps, res, post, pre)
    got_resid = bf16_dev_to_bits(out["resid"]).reshape(T, S, H)
    z_gpu = bf16_dev_to_bits(out["z"])
    if not mixed:
        np.testing.assert_array_equal(got_resid, ref["resid"])
        dz = np.abs(z_gpu.astype(np.int32) - ref["z"].astype(np.int32))
        assert dz.max() <= 1 and np.mean(dz == 0) > 0.99, (dz.max(), np.mean(dz == 0))
    else:
        check_mixed_epilogue(out, y_gpu, resid, gamma, eps, res, post, pre)
    q, s = oracle.mxfp8_quantize(oracle.bf16_bits_to_f64(z_gpu))
    np.testing.assert_array_equal(to_np(out["zq"]), q)
    np.testing.assert_array_equal(to_np(out["zs"]), s)
    # the whole chain against the oracle's own y
    get = oracle_experts(seed, E, H, I)
    y_ref = oracle.moe_step(x_bits, lg_np, k, get)["y"]
    chain = oracle.residual_norm_mxfp8(y_ref, resid, gamma, eps, res, post, pre)
    check_y(z_gpu, chain["z"])
    assert rel_fro(oracle.bf16_bits_to_f64(got_resid), oracle.bf16_bits_to_f64(chain["resid"])) <= 1e-2
    step.close()


def test_projection_and_epilogue_full_size_bs1():
    """Both fused steps at the bs1 shape (T=6, H=4096, E=256, k=8, I=2048):
    the logits, routing and epilogue everywhere, y on two sampled rows."""
    dev = torch.device("cuda", 0)
    T, H, E, k, I = 6, 4096, 256, 8, 2048
    seed = 42
    w = synthetic.make_weights(seed, E, H, I, 0, dev)
    x_bits = synth.x_bf16(seed, T, H)
    wr_bits = synth.router_weight_bf16(seed, E, H)
    resid, gamma, _ = _epilogue_inputs(seed, T, 1, H, False)
    step = MoEStep(H, I, E, k, w, T, 0)
    taps, tt = taps_for(T, k, E, H, I, 0, dev)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    out = step.forward_fused(dev_bf16(x_bits), w_router=dev_bf16(wr_bits), resid=dev_bf16(resid),
                             norm_weight=dev_bf16(gamma), rms_eps=1e-6, z_tap=True, taps=taps, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == abi.MOE_OK
    lg_gpu = to_np(out["logits"])
    lg_ref = oracle.router_logits(x_bits, wr_bits)
    err = np.abs(lg_gpu.astype(np.float64) - lg_ref)
    assert np.all(err <= logits_bound(x_bits, wr_bits) + np.abs(lg_ref) * 2.0 ** -24)
    t = {n: to_np(v) for n, v in tt.items()}
    check_routing_from_gpu_logits(t, lg_gpu, k, E)
    y_gpu = bf16_dev_to_bits(out["y"])
    ref = oracle.residual_norm_mxfp8(y_gpu, resid, gamma, 1e-6)
    np.testing.assert_array_equal(bf16_dev_to_bits(out["resid"]).reshape(T, 1, H), ref["resid"])
    z_gpu = bf16_dev_to_bits(out["z"])
    assert np.abs(z_gpu.astype(np.int32) - ref["z"].astype(np.int32)).max() <= 1
    q, s = oracle.mxfp8_quantize(oracle.bf16_bits_to_f64(z_gpu))
    np.testing.assert_array_equal(to_np(out["zq"]), q)
    np.testing.assert_array_equal(to_np(out["zs"]), s)
    rows = [0, 5]
    r = oracle.moe_step(x_bits, lg_gpu, k, oracle_experts(seed, E, H, I), rows=rows)
    check_y(y_gpu[rows], r["y"][rows])
    step.close()


def test_projection_and_epilogue_full_size_bs64_four_streams():
    """Both fused steps at the bs64 shape the bench times (T=384, H=4096, E=256
    + the shared expert, k=8, I=2048, four mixed residual streams): the
    tensor-core projection's logits and the routing everywhere, the epilogue
    everywhere, y on three sampled rows (first, middle, last)."""
    dev = torch.device("cuda", 0)
    T, H, E, k, I, S = 384, 4096, 256, 8, 2048, 4
    seed = 42
    w = synthetic.make_weights(seed, E, H, I, 1, dev)
    x_bits = synth.x_bf16(seed, T, H)
    wr_bits = synth.router_weight_bf16(seed, E, H)
    resid, gamma, (res, post, pre) = _epilogue_inputs(seed, T, S, H, True)
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    step = MoEStep(H, I, E, k, w, T, 1)
    taps, tt = taps_for(T, k, E, H, I, 1, dev)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    out = step.forward_fused(dev_bf16(x_bits), w_router=dev_bf16(wr_bits), resid=dev_bf16(resid),
                             norm_weight=dev_bf16(gamma), rms_eps=1e-6, mix_res=to_dev(res), mix_post=to_dev(post),
                             mix_pre=to_dev(pre), z_tap=True, taps=taps, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == abi.MOE_OK
    lg_gpu = to_np(out["logits"])
    lg_ref = oracle.router_logits(x_bits, wr_bits)
    err = np.abs(lg_gpu.astype(np.float64) - lg_ref)
    assert np.all(err <= logits_bound(x_bits, wr_bits) + np.abs(lg_ref) * 2.0 ** -24)
    t = {n: to_np(v) for n, v in tt.items()}
    ids = check_routing_from_gpu_logits(t, lg_gpu, k, E)
    # on rows whose top-k margins exceed twice the bound, the oracle's own logits choose the same experts
    safe = topk_margin(lg_ref, k) > 2 * logits_bound(x_bits, wr_bits).max(axis=1)
    assert safe.any()
    np.testing.assert_array_equal(ids[safe], oracle.topk_ids(lg_ref, k)[safe])
    y_gpu = bf16_dev_to_bits(out["y"])
    check_mixed_epilogue(out, y_gpu, resid, gamma, 1e-6, res, post, pre)
    z_gpu = bf16_dev_to_bits(out["z"])
    q, s_ = oracle.mxfp8_quantize(oracle.bf16_bits_to_f64(z_gpu))
    np.testing.assert_array_equal(to_np(out["zq"]), q)
    np.testing.assert_array_equal(to_np(out["zs"]), s_)
    rows = [0, T // 2, T - 1]
    sh = oracle.expert_weights_from_synth(seed, "shared", H, I)
    r = oracle.moe_step(x_bits, lg_gpu, k, oracle_experts(seed, E, H, I), shared=sh, rows=rows)
    check_y(y_gpu[rows], r["y"][rows])
    step.close()


def test_fused_argument_errors():
    dev = torch.device("cuda", 0)
    T, H, E, k, I = 4, 512, 8, 2, 256
    w = synthetic.make_weights(3, E, H, I, 0, dev)
    x = torch.zeros((T, H), dtype=torch.bfloat16, device=dev)
    lg = torch.zeros((T, E), dtype=torch.float32, device=dev)
    y = torch.zeros((T, H), dtype=torch.bfloat16, device=dev)
    resid = torch.zeros((T, 1, H), dtype=torch.bfloat16, device=dev)
    g = torch.ones((H,), dtype=torch.bfloat16, device=dev)
    zq = torch.zeros((T, H), dtype=torch.uint8, device=dev)
    zs = torch.zeros((T, H // 32), dtype=torch.uint8, device=dev)
    step = MoEStep(H, I, E, k, w, T, 0)
    call = lambda io, TT=T: abi.moe_forward_fused(step.plan, x, TT, io, y)
    assert call(abi.fused_io()) == abi.MOE_ERR_INVALID_ARG                       # no logits, no router weight
    assert call(None) == abi.MOE_ERR_INVALID_ARG
    assert call(abi.fused_io(logits=lg), T + 1) == abi.MOE_ERR_INVALID_ARG       # T > max_rows
    assert call(abi.fused_io(logits=lg), 0) == abi.MOE_OK                        # empty step
    ok = dict(logits=lg, num_streams=1, resid_in=resid, resid_out=resid, norm_weight=g, rms_eps=1e-6, zq=zq, zs=zs)
    assert call(abi.fused_io(**{**ok, "num_streams": 5})) == abi.MOE_ERR_INVALID_ARG
    assert call(abi.fused_io(**{**ok, "norm_weight": None})) == abi.MOE_ERR_INVALID_ARG
    assert call(abi.fused_io(**{**ok, "rms_eps": -1.0})) == abi.MOE_ERR_INVALID_ARG
    assert call(abi.fused_io(**{**ok, "rms_eps": float("nan")})) == abi.MOE_ERR_INVALID_ARG
    assert call(abi.fused_io(**{**ok, "zq": zq.data_ptr() + 8})) == abi.MOE_ERR_INVALID_ARG
    assert call(abi.fused_io(w_router=g.data_ptr() + 2)) == abi.MOE_ERR_INVALID_ARG  # misaligned router weight
    assert call(abi.fused_io(**ok)) == abi.MOE_OK
    torch.cuda.synchronize()
    step.close()
    gemv = MoEStep(H, I, E, k, w, T, 0, abi.MOE_FLAG_PATH_GEMV)
    assert abi.moe_forward_fused(gemv.plan, x, T, abi.fused_io(logits=lg), y) == abi.MOE_ERR_UNSUPPORTED
    gemv.close()
