"""Device-side row count and CUDA-graph replay (moe_forward_dev).

One step is captured in a CUDA graph once, with the row count read from device
memory. Replays with different row counts must each equal a step enqueued with
that count from the host (bit for bit: the same kernels, the same chunking),
and match the oracle. Rows at or past T must stay untouched. T = 0 is an empty
step, and an out-of-range count is clamped to max_rows and reported.
Source: "Beyond Day-0: Optimizing DeepSeek-V4.1 Flash in SGLang", section 3.1:
lengths are read from GPU memory, so a replayed CUDA graph uses the current length.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_top_gb300 import abi, synthetic
from moe_expert_layer_top_gb300.layer import MoEStep

from gpu_cases import bf16_dev_to_bits, check_y, oracle_experts

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import moe_expert_layer_top_gb300 as pkg
    pkg.build.build()
    abi.load()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("H,E,k,I,shared,tmax", [(512, 8, 2, 256, 0, 24), (512, 16, 4, 256, 1, 40)])
def test_graph_replay_with_device_row_count(H, E, k, I, shared, tmax):
    dev = torch.device("cuda", 0)
    seed = 11
    w = synthetic.make_weights(seed, E, H, I, shared, dev)
    x, lg, x_bits, lg_np = synthetic.make_inputs(seed, tmax, H, E, k, "zipf", dev)
    step = MoEStep(H, I, E, k, w, tmax, shared)
    d_T = torch.zeros(1, dtype=torch.int32, device=dev)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    y = torch.empty((tmax, H), dtype=torch.bfloat16, device=dev)

    # warm up outside the capture, then capture once
    d_T.fill_(tmax)
    step.forward_dev(x, lg, d_T, y, status)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.forward_dev(x, lg, d_T, y, status)
    torch.cuda.synchronize()

    get = oracle_experts(seed, E, H, I)
    sh = oracle.expert_weights_from_synth(seed, "shared", H, I) if shared else None
    for T in (tmax, 6, 1, 13, 0):
        y.fill_(float("nan"))
        status.fill_(-1)
        d_T.fill_(T)
        graph.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == abi.MOE_OK, (T, abi.moe_status_string(int(status.item())))
        got = bf16_dev_to_bits(y)
        assert np.all(np.isnan(y[T:].float().cpu().numpy())), f"rows past T={T} were written"
        if T == 0:
            continue
        y_host = step.forward(x[:T].contiguous(), lg[:T].contiguous())
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got[:T], bf16_dev_to_bits(y_host))
        r = oracle.moe_step(x_bits[:T], lg_np[:T], k, get, shared=sh)
        check_y(got[:T], r["y"])

    # a count past max_rows: clamped, reported, and the max_rows rows computed
    y.fill_(float("nan"))
    d_T.fill_(tmax + 5)
    graph.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == abi.MOE_ERR_DEVICE_BOUNDS
    assert not np.any(np.isnan(y.float().cpu().numpy()))
    step.close()


def test_forward_dev_argument_errors():
    dev = torch.device("cuda", 0)
    H, E, k, I, tmax = 512, 8, 2, 256, 8
    w = synthetic.make_weights(3, E, H, I, 0, dev)
    x = torch.zeros((tmax, H), dtype=torch.bfloat16, device=dev)
    lg = torch.zeros((tmax, E), dtype=torch.float32, device=dev)
    y = torch.zeros((tmax, H), dtype=torch.bfloat16, device=dev)
    d_T = torch.zeros(1, dtype=torch.int32, device=dev)
    step = MoEStep(H, I, E, k, w, tmax, 0)
    assert abi.moe_forward_dev(step.plan, x, lg, None, y) == abi.MOE_ERR_INVALID_ARG
    step.close()
    gemv = MoEStep(H, I, E, k, w, tmax, 0, abi.MOE_FLAG_PATH_GEMV)
    assert abi.moe_forward_dev(gemv.plan, x, lg, d_T, y) == abi.MOE_ERR_UNSUPPORTED
    gemv.close()


def test_graph_of_a_layer_stack():
    """Three layers in one captured graph, each layer's y the next layer's x
    (separate plans and weights). Inside the graph each route kernel follows
    the previous layer's expert kernel through a programmatic edge. Replays
    for several row counts equal the same three steps run one by one."""
    dev = torch.device("cuda", 0)
    H, E, k, I, tmax = 512, 8, 2, 256, 24
    layers = []
    for li in range(3):
        w = synthetic.make_weights(40 + li, E, H, I, 0, dev)
        layers.append((w, MoEStep(H, I, E, k, w, tmax, 0)))
    x, _, _, _ = synthetic.make_inputs(40, tmax, H, E, k, "zipf", dev)
    lgs = [synthetic.make_inputs(50 + li, tmax, H, E, k, "zipf", dev)[1] for li in range(3)]
    d_T = torch.full((1,), tmax, dtype=torch.int32, device=dev)
    ys = [torch.empty((tmax, H), dtype=torch.bfloat16, device=dev) for _ in range(3)]
    status = [torch.full((1,), -1, dtype=torch.int32, device=dev) for _ in range(3)]

    def stack():
        inp = x
        for li, (_, st) in enumerate(layers):
            st.forward_dev(inp, lgs[li], d_T, ys[li], status[li])
            inp = ys[li]
    stack()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        stack()
    torch.cuda.synchronize()
    for T in (tmax, 7, 1):
        for y in ys:
            y.fill_(float("nan"))
        d_T.fill_(T)
        graph.replay()
        torch.cuda.synchronize()
        assert all(int(s.item()) == abi.MOE_OK for s in status), T
        inp = x[:T].contiguous()
        for li, (_, st) in enumerate(layers):
            ref = st.forward(inp, lgs[li][:T].contiguous())
            torch.cuda.synchronize()
            np.testing.assert_array_equal(bf16_dev_to_bits(ys[li][:T]), bf16_dev_to_bits(ref))
            inp = ref
    for _, st in layers:
        st.close()
