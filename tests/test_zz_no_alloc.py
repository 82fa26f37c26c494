"""moe_forward_static_scratch: the MoE step for callers that cannot allocate.

Some callers cannot call cudaMalloc where they run the step. Examples are a
server whose allocator already owns nearly all device memory, code that must
not trigger cudaMalloc's synchronisation, and a plugin that is only handed its
buffers. For them the library keeps its scratch in a fixed device array.

This test calls that entry point through the C ABI, twice in a row. The two
calls share the array, and the second must not see leftovers of the first.
Both results are compared with the planned entry point's output (moe_forward),
within the tolerance of the other GPU tests. Oversized steps must be rejected.
The file sorts last, so a run that stops at the first failure has already run
every other test. It also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from moe_expert_layer_top_gb300 import abi, synthetic
from moe_expert_layer_top_gb300.layer import MoEStep

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


@pytest.mark.parametrize("T,H,E,k,I,routing,shared", [
    (6, 512, 8, 2, 256, "uniform", 0),
    (24, 4096, 64, 8, 2048, "uniform", 0),
    (20, 512, 8, 2, 256, "zipf", 1),
])
def test_static_scratch_matches_planned_forward_twice(T, H, E, k, I, routing, shared):
    dev = torch.device("cuda", 0)
    w = synthetic.make_weights(7, E, H, I, shared, dev)
    x, lg, _, _ = synthetic.make_inputs(7 + T, T, H, E, k, routing, dev)
    step = MoEStep(H, I, E, k, w, T, shared)
    y_ref = step.forward(x, lg)
    torch.cuda.synchronize()
    step.close()

    cfg = abi.MoeConfig(H, I, E, k, shared, 0, 0, 0)
    wabi = w.as_abi()
    st = torch.cuda.current_stream()
    for call in range(2):
        y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=dev)
        status = torch.full((1,), -1, dtype=torch.int32, device=dev)
        rc = abi.moe_forward_static_scratch(cfg, wabi, x, lg, T, y, status, st)
        assert rc == abi.MOE_OK, abi.moe_status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == abi.MOE_OK, call
        _close(y, y_ref)


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
