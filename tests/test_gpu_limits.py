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


def test_small_plan_after_large_plan_keeps_the_large_plan_working():
    """The route kernel's shared-memory limit is one setting per kernel for the
    whole process. A plan whose bitmap needs far more than the default (E = 256,
    max_rows = 2048: 64 KB of bitmap) must still run after a small plan is built."""
    T, H, E, k, I = 2048, 512, 256, 2, 256
    big = CudaStep(T, H, E, k, I, "zipf", seed=77)
    small = CudaStep(6, H, 8, 2, I, seed=78).run()
    assert small.status_code == abi.MOE_OK
    big.run()
    assert big.status_code == abi.MOE_OK, (abi.moe_status_string(big.status_code), big.diag)
    r = oracle.moe_step(big.x_bits, big.lg, k, oracle_experts(77, E, H, I), rows=[0, 1, T - 1])
    check_routing_bit_exact(big, r)
    check_y(big.y_bits[[0, 1, T - 1]], r["y"][[0, 1, T - 1]])
    small.close()
    big.close()
