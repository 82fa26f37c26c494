"""moe_forward_static_scratch: the MoE step for callers that cannot allocate.

Some callers cannot call cudaMalloc where they run the step. Examples are a
server whose allocator already owns nearly all device memory, code that must
not trigger cudaMalloc's synchronisation, and a plugin that is only handed its
buffers. For them the library keeps its scratch in a fixed device array.

This test calls that entry point through the C ABI, twice in a row, with a
larger step first and then a smaller one on other inputs: the two calls share
the array, and the second must not pick up leftovers of the first (ready
counts, combine counters, row lists, the placement ticket). Each result is
compared, within the tolerance of the other GPU tests, with the planned entry
point's output (moe_forward) on the same inputs and with the oracle over
every token row. Oversized steps must be rejected.
The file sorts last, so a run that stops at the first failure has already run
every other test. It also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from moe_expert_layer_top_gb300 import abi, synthetic
from moe_expert_layer_top_gb300.layer import MoEStep

from gpu_cases import check_y

pytestmark = pytest.mark.gpu

REL_FRO = 1e-2       # same tolerance as the oracle parity tests
MAX_ABS_RMS = 5e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    import moe_expert_layer_top_gb300.build as b
    b.build()
    abi.load()
    assert torch.cuda.is_available()


def _close(y, y_ref):
    a = y.float().cpu().numpy().astype(np.float64)
    r = y_ref.float().cpu().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(r ** 2)))
    fro = float(np.linalg.norm(a - r) / np.linalg.norm(r))
    assert fro <= REL_FRO, fro
    assert float(np.max(np.abs(a - r))) <= MAX_ABS_RMS * rms


CASES = [
    # H, E, k, I, shared, first call (T, routing, seed), second call (T, routing, seed)
    (512, 8, 2, 256, 0, (40, "zipf", 7), (6, "uniform", 8)),
    (1024, 16, 4, 512, 1, (48, "zipf", 9), (13, "uniform", 10)),
    (4096, 64, 8, 2048, 0, (24, "uniform", 11), (9, "zipf", 12)),
]


@pytest.mark.parametrize("H,E,k,I,shared,first,second", CASES,
                         ids=[f"H{c[0]}_E{c[1]}_k{c[2]}_sh{c[4]}" for c in CASES])
def test_static_scratch_two_calls_match_planned_forward_and_oracle(H, E, k, I, shared, first, second):
    from gpu_cases import full_oracle
    dev = torch.device("cuda", 0)
    wseed = 7
    w = synthetic.make_weights(wseed, E, H, I, shared, dev)
    cfg = abi.MoeConfig(H, I, E, k, shared, 0, 0, 0)
    wabi = w.as_abi()
    st = torch.cuda.current_stream()
    inputs, outs = {}, {}
    for call, (T, routing, seed) in enumerate((first, second)):
        x, lg, x_bits, lg_np = synthetic.make_inputs(seed, T, H, E, k, routing, dev)
        step = MoEStep(H, I, E, k, w, T, shared)
        y_ref = step.forward(x, lg)
        torch.cuda.synchronize()
        step.close()
        y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=dev)
        status = torch.full((1,), -1, dtype=torch.int32, device=dev)
        rc = abi.moe_forward_static_scratch(cfg, wabi, x, lg, T, y, status, st)
        assert rc == abi.MOE_OK, abi.moe_status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == abi.MOE_OK, call
        _close(y, y_ref)
        inputs[call] = (x_bits, lg_np, k, bool(shared))
        outs[call] = y.view(torch.int16).cpu().numpy().view(np.uint16)
    ref, _ = full_oracle(wseed, inputs, H, I)
    for call in outs:
        check_y(outs[call], ref[call]["y"])


def test_static_scratch_rejects_oversized_steps():
    dev = torch.device("cuda", 0)
    H, I, E, k = 4096, 2048, 8, 8
    w = synthetic.make_weights(3, E, H, I, 0, dev)
    cfg = abi.MoeConfig(H, I, E, k, 0, 0, 0, 0)
    T = 384  # about 59 MB of scratch at this shape, far over MOE_STATIC_SCRATCH_BYTES
    x = torch.zeros((T, H), dtype=torch.bfloat16, device=dev)
    lg = torch.zeros((T, E), dtype=torch.float32, device=dev)
    y = torch.zeros((T, H), dtype=torch.bfloat16, device=dev)
    assert abi.moe_forward_static_scratch(cfg, w.as_abi(), x, lg, T, y, None, None) == abi.MOE_ERR_UNSUPPORTED
    assert abi.moe_forward_static_scratch(cfg, w.as_abi(), x, lg, 0, y, None, None) == abi.MOE_OK
