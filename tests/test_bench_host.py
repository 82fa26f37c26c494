"""Host-side logic of bench.py that needs no GPU: the staleness check of the
committed ncu traffic record, and the traffic scaling that fills the bench
line's roofline.traffic."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_hash_ignores_comments_and_whitespace(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    c = tmp_path / "c.cu"
    a.write_text("int f(int x) {\n  return x + 1;  // one more\n}\n")
    b.write_text("/* a block\n   comment */\nint f(int x) {\n\n    return x + 1;\n}\n// trailing\n")
    c.write_text("int f(int x) {\n  return x + 2;  // one more\n}\n")
    assert bench.code_sha256(str(a)) == bench.code_sha256(str(b))
    assert bench.code_sha256(str(a)) != bench.code_sha256(str(c))


def test_committed_traffic_record_matches_the_expert_kernel():
    """The tensor-core kernel's record was taken on the code in the tree: the
    bench line then carries DRAM traffic scaled from it (1.0042 x the
    algorithmic bytes at capture), not null."""
    with open(os.path.join(ROOT, "profiles", "experts_mma_kernel_traffic.json")) as f:
        d = json.load(f)
    assert bench.kernel_code_sha256("mma") == d["source_code_sha256"]
    assert d["sources"] == [os.path.join("moe_expert_layer_top_gb300", "csrc", f) for f in bench.EXPERT_KERNELS["mma"][1]]
    algo = 1167851520  # bs1: 45 active experts x 3 x 2048 x 4096 x 33/32
    t = bench.traffic_per_launch(algo, "mma")
    ratio = (d["dram_bytes_read"] + d["dram_bytes_write"]) / d["algorithmic_bytes"]
    assert t == int(round(algo * ratio))
    assert 0.99 < t / algo < 1.02
