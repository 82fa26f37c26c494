"""Host-side logic of bench.py that needs no GPU: the staleness check of the
committed ncu traffic record, the traffic scaling that fills the bench
line's roofline.traffic, and the reference arm (the oracle on the host cores)
end to end on the tiny workload."""
import json
import os
import subprocess
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


def test_reference_arm_line():
    """bench.py --impl reference prints one JSON line: the oracle's step time
    as value, cpu_baseline and e2e describing the same run."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
           "--steps", "3", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "us/step" and d["higher_is_better"] is False
    assert d["steps"] == 3 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("tiny")
