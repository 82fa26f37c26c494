"""GPU parity at the limits the Guard accepts, on the default tensor-core path.

* T = max_rows = 4096: 128 bitmap words per expert and 128 routing blocks,
  then a last-block placement over every pair.
* E = 1024 and k = 32: the widest top-k (32 candidates per lane, 32 rounds).
* I = 16384: 128 K chunks per down unit and 256 gate/up blocks per expert.
* T = 4096, E = 256, k = 32 with the shared expert: about 17,000 tiles and
  4,400 chunks, the largest work lists the bitmap's shared-memory limit
  admits; the route kernel scans the tile and chunk counts packed in 16-bit
  halves of one integer, so the totals must stay below 2^15.
Routing, placement and x quantisation are compared with the oracle bit for
bit, and y within the stated tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_top_gb300 import abi

from gpu_cases import CudaStep, check_h_quantizer_bit_exact, check_routing_bit_exact, check_xquant_bit_exact, \
    check_y, oracle_experts

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import moe_expert_layer_top_gb300 as pkg
    pkg.build.build()
    abi.load()
    assert torch.cuda.is_available()


LIMITS = [
    # T, H, E, k, I, routing, shared
    (4096, 128, 8, 2, 128, "zipf", 1),      # the largest max_rows
    (8, 128, 1024, 32, 128, "uniform", 0),  # the most experts and the widest top-k
    (2, 128, 4, 2, 16384, "uniform", 1),    # the largest intermediate size
    (4096, 128, 256, 32, 128, "uniform", 1),  # the longest tile and chunk lists
]


@pytest.mark.parametrize("case", LIMITS, ids=[f"T{c[0]}_H{c[1]}_E{c[2]}_k{c[3]}_I{c[4]}" for c in LIMITS])
def test_parity_at_the_limits(case):
    T, H, E, k, I, routing, shared = case
    g = CudaStep(T, H, E, k, I, routing, shared, seed=90 + k).run()
    assert g.status_code == abi.MOE_OK, (abi.moe_status_string(g.status_code), g.diag)
    get = oracle_experts(90 + k, E, H, I)
    sh = oracle.expert_weights_from_synth(90 + k, "shared", H, I) if shared else None
    r = oracle.moe_step(g.x_bits, g.lg, k, get, shared=sh)
    check_routing_bit_exact(g, r)
    check_xquant_bit_exact(g, r)
    check_h_quantizer_bit_exact(g)
    check_y(g.y_bits, r["y"])
    g.close()
