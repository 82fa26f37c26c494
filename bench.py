"""Benchmark of the small-batch MXFP8 MoE step on GB300.

One step is one pass of the whole hot path over one batch of synthetic input:
route + place + quantise x, expert SwiGLU MLPs (gate/up, then down) with the combine fused into the expert kernel.

Default workload: the bs1 speculative-verify shape. That is T=6 token rows,
H=4096, E=256 routed experts, top-8, I=2048, MXFP8 weights (group-32 UE8M0
along K), uniform routing, seed 42.

The JSON line reports:
* value: microseconds per step, with inputs resident in HBM. There is no L2
  flush between steps: the step's active weights (0.8 to 1.9 GB) are far
  larger than the L2, and the timed steps cycle through 4 copies of the
  layer's weights at different addresses, so each step streams weights the
  previous 3 steps did not touch (a stack of identical layers). The time with
  an L2 flush before every step is reported beside it (detail.us_l2_flushed).
* roofline: the expert kernel's achieved HBM GB/s on the active experts'
  weight bytes, against the measured copy bandwidth.
* e2e: the same metric through the C ABI with host buffers (moe_forward_host).
* cpu_baseline: the oracle timed on the host cores on a bounded sample.
* also: the other row counts (24/96/384) as context.

--impl reference times the oracle instead: the plain CPU restatement of the
step, over every token row of each step at once (one process per row), so
ms_per_step x steps is the wall time of the timed steps.
Under torchrun each rank runs an independent replica. There is no collective
in the data path.
"""
from __future__ import annotations

import argparse
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "bs1"
SAMPLE_ROWS = 2        # oracle sample: this many token rows of the step, with every expert they touch
LAYER_COPIES = 4       # copies of the layer's weights the timed steps cycle through (no L2 flush)
ORACLE_WORKERS = 8     # spawn workers that prepare the oracle's weights (not timed)


# ----------------------------------------------------------------------------- oracle side (CPU)

def _oracle_expert(args):
    seed, e, H, I, fmt = args
    import oracle
    w = oracle.expert_weights_from_synth(seed, e, H, I, fmt=fmt)
    return e, w


def _oracle_prepare(seed, wl_name, rows, pool):
    import numpy as np  # noqa: F401
    import oracle
    import synth
    wl = synth.WORKLOADS[wl_name]
    x_bits = synth.x_bf16(seed, wl.T, wl.H)
    lg = synth.router_logits(seed, wl.T, wl.E, wl.k, wl.routing)
    ids = oracle.topk_ids(lg, wl.k)
    experts = sorted(set(int(e) for t in rows for e in ids[t]))
    jobs = [(seed, e, wl.H, wl.I, wl.fmt) for e in experts]
    if wl.shared:
        jobs.append((seed, "shared", wl.H, wl.I, wl.fmt))
    return x_bits, lg, experts, jobs


def _oracle_row_server(conn, seed: int, wl_name: str, t: int):
    """One token row of the step through the oracle, in its own process: draws
    the experts the row needs once, then computes the row on every request."""
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    os.environ["OMP_NUM_THREADS"] = "1"
    import oracle
    import synth
    wl = synth.WORKLOADS[wl_name]
    x = synth.x_bf16(seed, wl.T, wl.H)
    lg = synth.router_logits(seed, wl.T, wl.E, wl.k, wl.routing)
    w = {int(e): oracle.expert_weights_from_synth(seed, int(e), wl.H, wl.I, fmt=wl.fmt)
         for e in oracle.topk_ids(lg[t:t + 1], wl.k)[0]}
    sh = oracle.expert_weights_from_synth(seed, "shared", wl.H, wl.I, fmt=wl.fmt) if wl.shared else None
    conn.send("ready")
    while conn.recv() is not None:
        r = oracle.moe_step(x, lg, wl.k, w, shared=sh, rows=[t], swiglu_limit=wl.swiglu_limit)
        conn.send(r["y"][t])


def oracle_all_cores(seed: int, wl_name: str, steps: int, check_rows: dict | None = None, warmup: int = 0):
    """The oracle over every token row of the step at once, one persistent
    spawned process per row: the wall time of whole steps. `warmup` steps run
    first and are not timed. The rows must equal the single-thread run's
    (check_rows: row -> y bits), when given."""
    import numpy as np
    import synth
    wl = synth.WORKLOADS[wl_name]
    if wl.T > (os.cpu_count() or 1):
        raise RuntimeError("more token rows than host cores")
    ctx = mp.get_context("spawn")
    conns, procs = [], []
    try:
        for t in range(wl.T):
            a, b = ctx.Pipe()
            p = ctx.Process(target=_oracle_row_server, args=(b, seed, wl_name, t), daemon=True)
            p.start()
            conns.append(a)
            procs.append(p)
        for c in conns:
            if c.recv() != "ready":
                raise RuntimeError("row process failed")
        times, got = [], {}
        for i in range(warmup + steps):
            t0 = time.perf_counter()
            for c in conns:
                c.send(1)
            got = {t: c.recv() for t, c in enumerate(conns)}
            if i >= warmup:
                times.append(time.perf_counter() - t0)
    finally:
        for c in conns:
            try:
                c.send(None)
            except (BrokenPipeError, OSError):
                pass
        for p in procs:
            p.join(timeout=30)
    for t, y in (check_rows or {}).items():
        if not np.array_equal(got[t], y):
            raise RuntimeError(f"all-cores oracle row {t} differs from the single-thread run")
    return {"us_per_step": statistics.median(times) * 1e6, "us_mean": statistics.mean(times) * 1e6,
            "cores": wl.T, "steps": steps, "warmup": warmup}


def oracle_baseline(seed: int, wl_name: str, steps: int, warmup: int, result_q, gpu_done=None,
                    with_all_cores=True):
    """Runs in a spawned process: times the oracle on a bounded sample of the workload."""
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    import oracle
    import synth
    wl = synth.WORKLOADS[wl_name]
    rows = list(range(min(SAMPLE_ROWS, wl.T)))
    ctx = mp.get_context("spawn")
    with ctx.Pool(ORACLE_WORKERS) as pool:
        x_bits, lg, experts, jobs = _oracle_prepare(seed, wl_name, rows, pool)
        got = dict(pool.map(_oracle_expert, jobs))
    shared = got.pop("shared", None)
    times = []
    for i in range(warmup + steps):
        t0 = time.perf_counter()
        r = oracle.moe_step(x_bits, lg, wl.k, got, shared=shared, rows=rows, swiglu_limit=wl.swiglu_limit)
        dt = time.perf_counter() - t0
        if i >= warmup:
            times.append(dt)
    per_sample = statistics.median(times)
    scale = wl.T / len(rows)
    all_cores = None
    # every row at once, one process per row: the whole step's wall time. It
    # uses many host cores, so it waits until the GPU timing is over.
    if gpu_done is not None:
        gpu_done.wait(timeout=600)
    if with_all_cores and wl.T <= 64:
        try:
            all_cores = oracle_all_cores(seed, wl_name, 3, {t: r["y"][t] for t in rows})
        except Exception as exc:  # reported, not fatal: the single-thread baseline stands
            all_cores = {"error": str(exc)[:200]}
    result_q.put({
        "us_per_step": per_sample * scale * 1e6,
        "sample_s": per_sample,
        "rows": len(rows),
        "experts": len(experts) + (1 if shared is not None else 0),
        "scale": scale,
        "steps": steps,
        "cores": 1,
        "all_cores": all_cores,
    })


def bench_config(wl, args, world: int) -> dict:
    """The workload and the timing policy, printed the same way by both arms."""
    l2 = ("flushed before every step (memset of a buffer >= 2x L2, outside the timed events)"
          if args.l2 == "flush" else
          f"inputs larger than L2: no flush; steps cycle through {args.layer_copies} copies of the layer's "
          f"weights (a stack of identical layers), so every step streams active expert weights that the last "
          f"{args.layer_copies - 1} steps did not touch; the kernels' code and the step's small inputs stay in L2")
    return {
        "workload": f"{wl.name}: T={wl.T} token rows, H={wl.H}, E={wl.E}, top-{wl.k}, I={wl.I}, "
                    f"shared={wl.shared}, routing={wl.routing}, weights={wl.fmt}",
        "T": wl.T, "H": wl.H, "E": wl.E, "top_k": wl.k, "I": wl.I, "shared": wl.shared, "routing": wl.routing,
        "weights": wl.fmt, "swiglu_limit": wl.swiglu_limit, "seed": args.seed, "l2": l2,
        "parallelism": "replicas" if world > 1 else "single GPU",
    }


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, out_path: str | None):
        self.proc = None
        self.out_path = out_path
        self.gpu_index = gpu_index
        try:
            self.f = open(out_path, "w") if out_path else subprocess.DEVNULL
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "power": float(parts[3]),
                             "hw_slowdown": parts[5], "hw_thermal": parts[6], "sw_thermal": parts[7],
                             "sw_power_cap": parts[8]})
            except ValueError:
                continue
        if self.out_path:
            with open(self.out_path, "w") as f:
                f.write(out)
        return rows


def summarise_clocks(rows):
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
    loaded = [r for r in rows if r["power"] > 200] or rows
    reasons = set()
    for r in loaded:
        for key, name in (("hw_slowdown", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                          ("sw_thermal", "sw_thermal_slowdown"), ("sw_power_cap", "sw_power_cap")):
            if r[key].lower() == "active":
                reasons.add(name)
    return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": max(r["max"] for r in rows),
            "reasons": sorted(reasons), "samples": len(loaded)}


# ----------------------------------------------------------------------------- GPU side

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


EXPERT_KERNELS = {
    # path -> (kernel, source files of its device code, committed ncu traffic summary)
    "gemv": ("experts_kernel (persistent CUDA-core gate/up + down GEMV)",
             ("experts.cu", "combine.cuh", "device.cuh"), "experts_kernel_traffic.json"),
    "mma": ("experts_mma_kernel (persistent tcgen05 block-scaled MXFP8 MMA)",
            ("experts_mma.cu", "combine.cuh", "device.cuh"), "experts_mma_kernel_traffic.json"),
}
PATH_FLAGS = {"auto": 0, "gemv": 1 << 1, "mma": 1 << 2}
MMA_MIN_ROWS = 1  # the library's default: the tensor-core kernel at every row count


def kernel_path(path, T):
    if path != "auto":
        return path
    return "mma" if T >= MMA_MIN_ROWS else "gemv"


def code_sha256(*paths):
    """sha256 of C++/CUDA sources (in the given order) with comments and
    whitespace removed: the hash changes when the code does, not when a
    comment does."""
    import hashlib
    import re
    parts = []
    for path in paths:
        with open(path) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        parts.append("".join(text.split()))
    return hashlib.sha256("\n".join(parts).encode()).hexdigest()


def kernel_code_sha256(path="mma"):
    """code_sha256 of the device sources an expert kernel is compiled from."""
    return code_sha256(*(os.path.join(ROOT, "moe_expert_layer_top_gb300", "csrc", f) for f in EXPERT_KERNELS[path][1]))


def traffic_per_launch(algorithmic_bytes, path="gemv"):
    """DRAM bytes per expert-kernel launch from the committed ncu capture, scaled
    by the active weight bytes; None if the kernel's code changed since then."""
    summary = EXPERT_KERNELS[path][2]
    p = os.path.join(ROOT, "profiles", summary)
    try:
        with open(p) as f:
            d = json.load(f)
        sha = kernel_code_sha256(path)
    except OSError:
        return None
    if sha != d.get("source_code_sha256"):
        return None
    ratio = (d["dram_bytes_read"] + d["dram_bytes_write"]) / d["algorithmic_bytes"]
    return int(round(algorithmic_bytes * ratio))


def active_experts(lg, k, shared):
    import numpy as np
    ids = np.argsort(-lg, axis=1, kind="stable")[:, :k]
    return len(set(ids.ravel().tolist())) + (1 if shared else 0)


def flush(buf):
    """Evict L2 before a step by writing a buffer of twice its size (buf None: no flush)."""
    if buf is not None:
        buf.zero_()


def lead_in(stream, us=200):
    """A GPU spin of about `us` microseconds, enqueued after the synchronize and
    before the first timed event: the host then enqueues the first timed steps
    while the GPU is still busy, so no step's events include the host's launch
    latency. It runs before the timed region and is not one of the step's kernels."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(us * 2000))  # cycles, at about 2 GHz


def time_gpu_workload(wl, weight_sets, steps, warmup, flush_buf, seed, flags=0):
    """Times `steps` steps, then, in a second pass with the plans' kernel timing
    on, the expert kernel alone. Kernel timing records events between the two
    launches, which would break their programmatic-dependent-launch overlap,
    so the step times come from plans without it.
    weight_sets: one or more copies of the layer's weights at different
    addresses, one plan each; steps alternate between them. With no flush this
    is a stack of identical layers: every step streams weights that the
    previous step did not touch, while the kernels' code and the small inputs
    stay in L2. flush_buf (or None) evicts L2 before every step instead."""
    import torch
    from moe_expert_layer_top_gb300 import abi, synthetic
    from moe_expert_layer_top_gb300.layer import MoEStep, MoEWeightsMXFP8

    def routed(w):
        return w if wl.shared else MoEWeightsMXFP8(w.w_gate, w.s_gate, w.w_up, w.s_up, w.w_down, w.s_down)
    ws = [routed(w) for w in weight_sets]
    x, lg, _, lg_np = synthetic.make_inputs(seed, wl.T, wl.H, wl.E, wl.k, wl.routing)
    wfmt = abi.MOE_WEIGHTS_MXFP4 if wl.fmt == "mxfp4" else abi.MOE_WEIGHTS_MXFP8
    steps_ = [MoEStep(wl.H, wl.I, wl.E, wl.k, w, wl.T, wl.shared, flags=flags, weight_format=wfmt,
                      swiglu_limit=wl.swiglu_limit) for w in ws]
    y = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    # one device status word per step: every step must finish with MOE_OK
    st_words = torch.full((warmup + steps,), -1, dtype=torch.int32, device="cuda")
    for i in range(warmup):
        flush(flush_buf)
        steps_[i % len(steps_)].forward(x, lg, y=y, d_status=st_words[i:i + 1])
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    lead_in(stream)
    for i in range(steps):
        flush(flush_buf)
        starts[i].record(stream)
        steps_[(warmup + i) % len(steps_)].forward(x, lg, y=y, d_status=st_words[warmup + i:warmup + i + 1])
        ends[i].record(stream)
    torch.cuda.synchronize()
    per_step = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    # the same steps back to back, one event pair around all of them: consecutive
    # steps overlap through programmatic dependent launch, as layers of a model would
    b2b = None
    if flush_buf is None:
        a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        lead_in(stream)
        a_ev.record(stream)
        for i in range(steps):
            steps_[(warmup + i) % len(steps_)].forward(x, lg, y=y)
        b_ev.record(stream)
        torch.cuda.synchronize()
        b2b = a_ev.elapsed_time(b_ev) / steps
    words = st_words.cpu().tolist()
    bad = [(i, w) for i, w in enumerate(words) if w != abi.MOE_OK]
    status = 0 if not bad else bad[0][1]
    if bad:
        print(f"warning: {len(bad)} of {len(words)} steps reported a device status: first {bad[0]}, "
              f"diagnostics {steps_[0].diagnostics()}", file=sys.stderr)
    # second pass: the expert kernel's own duration (CUDA events on the launch stream)
    ksteps = [MoEStep(wl.H, wl.I, wl.E, wl.k, w, wl.T, wl.shared, flags=abi.MOE_FLAG_TIMING | flags,
                      weight_format=wfmt, swiglu_limit=wl.swiglu_limit) for w in ws]
    for i in range(max(3, warmup // 2)):
        flush(flush_buf)
        ksteps[i % len(ksteps)].forward(x, lg, y=y)
    torch.cuda.synchronize()
    for k in ksteps:
        k.kernel_times()
    for i in range(steps):
        flush(flush_buf)
        ksteps[i % len(ksteps)].forward(x, lg, y=y)
    expert_ms, launches = 0.0, 0
    for k in ksteps:
        m_, n_ = k.kernel_times()
        expert_ms += m_
        launches += n_
        k.close()
    for s_ in steps_[1:]:
        s_.close()
    A = active_experts(lg_np, wl.k, wl.shared)
    weight_bytes = A * wl.expert_bytes
    step_bytes = weight_bytes + wl.T * wl.H * 2 + wl.T * wl.E * 4 + wl.T * wl.H * 2
    res = {
        "ms_steps": per_step,
        "ms_back_to_back": b2b,
        "ms_mean": sum(per_step) / len(per_step),
        "ms_median": statistics.median(per_step),
        "ms_min": min(per_step),
        "ms_max": max(per_step),
        "expert_ms_mean": expert_ms / max(launches, 1),
        "expert_launches": launches,
        "active_experts": A,
        "weight_bytes": weight_bytes,
        "step_bytes": step_bytes,
        "status": status,
        "bad_steps": len(bad),
        "step": steps_[0],
        "x": x,
        "lg": lg,
    }
    return res


def time_fused_workload(wl, weight_sets, steps, warmup, flush_buf, seed, n_streams):
    """Times moe_forward_fused three ways on the same routing. Buffers are
    allocated once.
    * "full": the router projection from a bf16 W_r [E][H] in front, and
      n_streams residual streams behind (mixing coefficients when more than
      one) with RMSNorm + MXFP8.
    * "projection": the router projection alone.
    * "plain": the plain step on the logits that the projection produced.
    The differences are the cost of each fused step."""
    import numpy as np
    import torch
    import synth
    from moe_expert_layer_top_gb300 import abi
    from moe_expert_layer_top_gb300.layer import MoEStep, MoEWeightsMXFP8
    wfmt = abi.MOE_WEIGHTS_MXFP4 if wl.fmt == "mxfp4" else abi.MOE_WEIGHTS_MXFP8
    plans = []
    for weights in weight_sets:  # steps alternate between the copies, as in time_gpu_workload
        w = weights if wl.shared else MoEWeightsMXFP8(weights.w_gate, weights.s_gate, weights.w_up, weights.s_up,
                                                      weights.w_down, weights.s_down)
        plans.append(MoEStep(wl.H, wl.I, wl.E, wl.k, w, wl.T, wl.shared, weight_format=wfmt,
                             swiglu_limit=wl.swiglu_limit))
    step = plans[0]
    bf = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16).copy()).view(torch.bfloat16).cuda()
    T, H, S = wl.T, wl.H, n_streams
    x = bf(synth.x_bf16(seed, T, H))
    wr = bf(synth.router_weight_bf16(seed, wl.E, H))
    resid = bf(synth.residual_bf16(seed, T, S, H))
    gamma = bf(synth.norm_weight_bf16(seed, H))
    coef = [None, None, None]
    if S > 1:
        coef = [torch.from_numpy(c).cuda() for c in synth.mix_coefficients(seed, T, S)]
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    logits = torch.empty((T, wl.E), dtype=torch.float32, device="cuda")
    logits_in = torch.empty_like(logits)
    resid_out = torch.empty_like(resid)
    zq = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    zs = torch.empty((T, H // 32), dtype=torch.uint8, device="cuda")
    ios = {
        "full": abi.fused_io(w_router=wr, logits=logits, num_streams=S, resid_in=resid, resid_out=resid_out,
                             mix_res=coef[0], mix_post=coef[1], mix_pre=coef[2], norm_weight=gamma, rms_eps=1e-6,
                             zq=zq, zs=zs),
        "projection": abi.fused_io(w_router=wr, logits=logits),
        "plain": abi.fused_io(logits=logits_in),
    }
    stream = torch.cuda.current_stream()
    abi.check("moe_forward_fused", abi.moe_forward_fused(step.plan, x, T, ios["projection"], y, None, None, stream))
    torch.cuda.synchronize()
    logits_in.copy_(logits)
    active = active_experts(logits.cpu().numpy(), wl.k, wl.shared)
    out = {"active_experts": active, "extra_bytes": wl.E * H * 2 + 2 * T * S * H * 2 + H * 2 + T * H + T * H // 32}
    bad = []
    for name, io in ios.items():
        st_words = torch.full((warmup + steps,), -1, dtype=torch.int32, device="cuda")
        for i in range(warmup):
            flush(flush_buf)
            abi.check("moe_forward_fused", abi.moe_forward_fused(plans[i % len(plans)].plan, x, T, io, y, None,
                                                                 st_words[i:i + 1], stream))
        torch.cuda.synchronize()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        lead_in(stream)
        for i in range(steps):
            flush(flush_buf)
            starts[i].record(stream)
            abi.moe_forward_fused(plans[(warmup + i) % len(plans)].plan, x, T, io, y, None,
                                  st_words[warmup + i:warmup + i + 1], stream)
            ends[i].record(stream)
        torch.cuda.synchronize()
        per_step = [a.elapsed_time(b) for a, b in zip(starts, ends)]
        bad += [v for v in st_words.cpu().tolist() if v != abi.MOE_OK]
        out[name] = {"ms_mean": sum(per_step) / len(per_step), "ms_median": statistics.median(per_step)}
    for p_ in plans:
        p_.close()
    out["ms_mean"], out["ms_median"] = out["full"]["ms_mean"], out["full"]["ms_median"]
    out["status"] = bad[0] if bad else 0
    return out


def mxfp8_tensor_peak():
    """Dense block-scaled MXFP8 MMA peak (TFLOP/s): the measured bf16 GEMM burst
    figure times the nominal fp8 / bf16 ratio (4.5 / 2.25)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return 2.0 * float(json.load(f)["bf16_tflops"]), "measured bf16 burst x 2 (nominal fp8/bf16 ratio)"
    return 2.0 * 1900.0, "fallback bf16 x 2"


def step_flops(wl):
    """Algorithmic flops of the expert GEMMs of one step: 2 * (T*k + T*shared) * 3 * H * I."""
    return 2 * (wl.T * wl.k + wl.T * wl.shared) * 3 * wl.H * wl.I


def time_l2_warm_graph(step, x, lg, wl, steps):
    """Secondary figure: one step captured in a CUDA graph (moe_forward_dev with
    the row count on the device), replayed back to back with no L2 flush."""
    import torch
    d_T = torch.full((1,), wl.T, dtype=torch.int32, device="cuda")
    y = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step.forward_dev(x, lg, d_T, y, status)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step.forward_dev(x, lg, d_T, y, status)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        lead_in(s)
        a.record(s)
        for _ in range(steps):
            g.replay()
        b.record(s)
        torch.cuda.synchronize()
    return {"us_per_step": round(a.elapsed_time(b) * 1e3 / steps, 3), "status": int(status.item()),
            "how": f"one step captured in a CUDA graph (device-side row count), replayed {steps} times back to "
                   "back with no L2 flush"}


def input_checksums(wl, weights, seed):
    """Fingerprints of the step's synthetic inputs, so a run can be matched to
    its inputs: sha256 of the token rows' and logits' bytes (host), and the
    wrapping sum of each weight tensor's 64-bit words (device)."""
    import hashlib
    import synth
    x = synth.x_bf16(seed, wl.T, wl.H)
    lg = synth.router_logits(seed, wl.T, wl.E, wl.k, wl.routing)
    out = {"x_sha256": hashlib.sha256(x.tobytes()).hexdigest()[:16],
           "logits_sha256": hashlib.sha256(lg.tobytes()).hexdigest()[:16]}
    import torch
    for name in ("w_gate", "s_gate", "w_up", "s_up", "w_down", "s_down"):
        t = getattr(weights, name)
        n = t.numel() // 8 * 8
        out[name + "_sum64"] = int(t.reshape(-1)[:n].view(torch.int64).sum().item()) & ((1 << 64) - 1)
    return out


def time_e2e(step, wl, seed, steps, warmup):
    """moe_forward_host: pinned host x/logits in, host y out, copies inside the timed region."""
    import numpy as np
    import torch
    import synth
    from moe_expert_layer_top_gb300 import abi
    xh = torch.from_numpy(synth.x_bf16(seed, wl.T, wl.H).view(np.int16).copy()).pin_memory()
    lh = torch.from_numpy(synth.router_logits(seed, wl.T, wl.E, wl.k, wl.routing)).pin_memory()
    yh = torch.empty((wl.T, wl.H), dtype=torch.int16).pin_memory()
    for _ in range(warmup):
        assert step.forward_host(xh, lh, yh) == abi.MOE_OK
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        st = step.forward_host(xh, lh, yh)
        times.append(time.perf_counter() - t0)
        assert st == abi.MOE_OK
    h2d = wl.T * wl.H * 2 + wl.T * wl.E * 4
    d2h = wl.T * wl.H * 2 + 4
    return {"value": statistics.mean(times) * 1e6, "unit": "us/step", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "median_us": statistics.median(times) * 1e6}


def max_over_ranks(values, world, device):
    """Element-wise max of per-rank values over the process group (the slowest
    replica sets the step time). One rank: the values themselves."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def run_gpu(args):
    import torch
    import torch.distributed as dist
    import synth
    from moe_expert_layer_top_gb300 import build as _build
    from moe_expert_layer_top_gb300 import synthetic

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    seed = args.seed
    wl = synth.WORKLOADS[args.workload]
    if args.experts:
        import dataclasses
        wl = dataclasses.replace(wl, E=args.experts, name=f"{wl.name}-E{args.experts}")
        args.no_cpu_baseline = args.no_others = True
    if args.fused:
        args.no_cpu_baseline = True

    # The oracle's worker pool is spawned before the first GPU call.
    cpu_q = None
    cpu_proc = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ctx = mp.get_context("spawn")
        cpu_q = ctx.Queue()
        gpu_done = ctx.Event()
        cpu_proc = ctx.Process(target=oracle_baseline, args=(seed, args.workload, 3, 1, cpu_q, gpu_done))
        cpu_proc.start()

    _build.build()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev_props = torch.cuda.get_device_properties(local)
    l2 = getattr(dev_props, "L2_cache_size", 128 << 20)
    flush_buf = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device="cuda")

    _wcache = {}

    def weights_for(w_l):
        """Synthetic weights of a workload's format and shape (with the shared expert), made once."""
        key = (w_l.fmt, w_l.E, w_l.H, w_l.I)
        if key not in _wcache:
            _wcache[key] = synthetic.make_weights(seed, w_l.E, w_l.H, w_l.I, shared=1, fmt=w_l.fmt)
            torch.cuda.synchronize()
        return _wcache[key]

    weights = weights_for(wl)

    _wcopies = {}

    def weight_sets_for(w_l):
        """LAYER_COPIES copies of a layer's weights at different addresses (see
        time_gpu_workload). Four: the copies' scale bytes, which the kernel reads
        at normal L2 priority, then exceed the L2 together (at bs1 about 4 x 35 MB)."""
        key = (w_l.fmt, w_l.E, w_l.H, w_l.I)
        if key not in _wcopies:
            from moe_expert_layer_top_gb300.layer import MoEWeightsMXFP8
            w0 = weights_for(w_l)
            sets = [w0]
            for _ in range(args.layer_copies - 1):
                sets.append(MoEWeightsMXFP8(*[None if getattr(w0, f) is None else getattr(w0, f).clone()
                                              for f in MoEWeightsMXFP8.__dataclass_fields__]))
            torch.cuda.synchronize()
            _wcopies[key] = sets
        return _wcopies[key]

    clocks = ClockSampler(local, args.clocks_log)
    time.sleep(0.05)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    flags = PATH_FLAGS[args.path]
    # L2 between timed steps. "inputs" (default): no flush; every step streams its active
    # weights (about 9x the L2 at bs1) from HBM, and the kernels' code and the step's
    # small inputs stay in L2, as they would across a model's layers. "flush": L2 is
    # evicted before every step (outside the timed events). The other policy is also
    # timed on the main workload and reported beside the value.
    main_flush = flush_buf if args.l2 == "flush" else None
    other_flush = None if args.l2 == "flush" else flush_buf
    if args.fused:
        r = time_fused_workload(wl, weight_sets_for(wl), args.steps, args.warmup, main_flush, seed, args.fused)
        clocks.stop()
        if rank == 0:
            print(json.dumps({"metric": "fused MoE step us (router projection + residual streams + RMSNorm + MXFP8)",
                              "workload": wl.name, "streams": args.fused, "value": round(r["ms_mean"] * 1e3, 3),
                              "unit": "us/step", "us_median": round(r["ms_median"] * 1e3, 3),
                              "us_projection_only": round(r["projection"]["ms_mean"] * 1e3, 3),
                              "us_same_routing_plain": round(r["plain"]["ms_mean"] * 1e3, 3),
                              "active_experts": r["active_experts"],
                              "status": r["status"], "steps": args.steps, "warmup": args.warmup}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return
    main = time_gpu_workload(wl, weight_sets_for(wl), args.steps, args.warmup, main_flush, seed, flags)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clock_rows = clocks.stop()

    ms, exp_ms = max_over_ranks([main["ms_mean"], main["expert_ms_mean"]], world, "cuda")

    other = time_gpu_workload(wl, weight_sets_for(wl), max(args.steps // 2, 5), max(args.warmup, 3), other_flush,
                              seed, flags)
    other["step"].close()
    e2e = None if args.no_e2e else time_e2e(main["step"], wl, seed, max(args.steps, 10), 3)
    l2_warm = None
    if kernel_path(args.path, wl.T) == "mma" and world == 1:
        l2_warm = time_l2_warm_graph(main["step"], main["x"], main["lg"], wl, max(args.steps, 10))

    also = {}
    if not args.no_others and world == 1:
        others = ["bs4", "bs16", "bs64"]
        if flags != PATH_FLAGS["gemv"]:
            others += ["bs1_fp4", "bs4_fp4", "bs64_fp4"]  # MXFP4: tensor-core kernel only
        tpeak, _ = mxfp8_tensor_peak()
        for name in others:
            if name == wl.name:
                continue
            o = synth.WORKLOADS[name]
            r = time_gpu_workload(o, weight_sets_for(o), max(args.steps // 2, 5), max(args.warmup, 3), main_flush, seed,
                                  flags)
            peak, _ = measured_peaks()
            also[name] = {"T": o.T, "I": o.I, "weights": o.fmt, "swiglu_limit": o.swiglu_limit,
                          "expert_kernel": kernel_path(args.path, o.T),
                          "us_per_step": round(r["ms_mean"] * 1e3, 2),
                          "us_median": round(r["ms_median"] * 1e3, 2),
                          "expert_kernel_us": round(r["expert_ms_mean"] * 1e3, 2),
                          "active_experts": r["active_experts"],
                          "expert_gbs": round(r["weight_bytes"] / (r["expert_ms_mean"] * 1e-3) / 1e9, 1),
                          "expert_frac": round(r["weight_bytes"] / (r["expert_ms_mean"] * 1e-3) / 1e9 / peak, 3),
                          "tensor_tflops": round(step_flops(o) / (r["expert_ms_mean"] * 1e-3) / 1e12, 1),
                          "tensor_frac": round(step_flops(o) / (r["expert_ms_mean"] * 1e-3) / 1e12 / tpeak, 4),
                          "status": r["status"]}
            r["step"].close()
        # the steps either side, fused: router projection + residual streams + RMSNorm + MXFP8
        if flags != PATH_FLAGS["gemv"]:
            for base, S in (("bs1", 1), ("bs64", 4)):
                o = synth.WORKLOADS[base]
                r = time_fused_workload(o, weight_sets_for(o), max(args.steps // 2, 5), max(args.warmup, 3), main_flush,
                                        seed, S)
                us = {n: r[n]["ms_mean"] * 1e3 for n in ("full", "projection", "plain")}
                also[f"{base}_fused_s{S}"] = {
                    "T": o.T, "streams": S, "router_projection": f"bf16 W_r [{o.E}][{o.H}]",
                    "active_experts": r["active_experts"],
                    "us_per_step": round(us["full"], 2), "us_median": round(r["ms_median"] * 1e3, 2),
                    "us_same_routing_plain": round(us["plain"], 2),
                    "us_projection_only": round(us["projection"], 2),
                    "projection_us": round(us["projection"] - us["plain"], 2),
                    "epilogue_us": round(us["full"] - us["projection"], 2),
                    "extra_bytes": r["extra_bytes"], "status": r["status"]}

    if rank != 0:
        main["step"].close()
        if world > 1:
            dist.destroy_process_group()
        return

    cpu = None
    if cpu_q is not None:
        gpu_done.set()  # the GPU timing is over: the oracle may use every host core now
        cpu = cpu_q.get(timeout=900)
        cpu_proc.join(timeout=60)

    peak, peak_kind = measured_peaks()
    achieved = main["weight_bytes"] / (exp_ms * 1e-3) / 1e9
    path = kernel_path(args.path, wl.T)
    line = {
        "metric": "MoE step us & achieved HBM GB/s (% of roofline) at 6/24/96/384 token rows",
        "value": round(ms * 1e3, 3),
        "unit": "us/step",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3xe4m3->f32 (MXFP8 weights and activations, bf16 in/out)",
        "data": "synthetic (seeded counter-based generator; random-init weights, MXFP8-quantised on device)",
        "config": bench_config(wl, args, world),
        "detail": {
            "expert_kernel": path,
            "active_experts": main["active_experts"],
            "step_bytes": main["step_bytes"],
            "step_gbs": round(main["step_bytes"] / (ms * 1e-3) / 1e9, 1),
            "us_median": round(main["ms_median"] * 1e3, 3),
            "us_min": round(main["ms_min"] * 1e3, 3),
            "us_max": round(main["ms_max"] * 1e3, 3),
            "us_back_to_back": None if main["ms_back_to_back"] is None else round(main["ms_back_to_back"] * 1e3, 3),
            "active_weight_mb": round(main["weight_bytes"] / 1e6, 1),
            "l2_mb": round(l2 / 1e6, 1),
            ("us_l2_flushed" if args.l2 != "flush" else "us_no_flush"): round(other["ms_mean"] * 1e3, 3),
            ("expert_kernel_us_l2_flushed" if args.l2 != "flush" else "expert_kernel_us_no_flush"):
                round(other["expert_ms_mean"] * 1e3, 3),
            "status": main["status"],
            "steps_with_device_error": main["bad_steps"],
            "inputs": input_checksums(wl, weights, seed),
        },
        "roofline": {
            "bound": "hbm",
            "kernel": EXPERT_KERNELS[path][0],
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic_per_launch(main["weight_bytes"], path),
            "traffic_source": f"profiles/{EXPERT_KERNELS[path][2]} (ncu capture, scaled by weight bytes)",
            "algorithmic_bytes_per_launch": main["weight_bytes"],
            "kernel_us": round(exp_ms * 1e3, 3),
        },
        "e2e": e2e,
        "l2_warm": l2_warm,
        "tensor": {"tflops": round(step_flops(wl) / (exp_ms * 1e-3) / 1e12, 2),
                   "peak": round(mxfp8_tensor_peak()[0], 1), "peak_kind": mxfp8_tensor_peak()[1],
                   "frac": round(step_flops(wl) / (exp_ms * 1e-3) / 1e12 / mxfp8_tensor_peak()[0], 5),
                   "flops_per_step": step_flops(wl),
                   "note": "expert GEMM flops 2*(T*k + T*shared)*3*H*I over the expert kernel time; the step is "
                           "bound by HBM at this row count"},
        "gpu_launches": 2 * args.steps,
        "clocks": summarise_clocks(clock_rows),
    }
    if cpu is not None:
        line["cpu_baseline"] = {
            "value": round(cpu["us_per_step"], 1), "unit": "us/step", "cores": cpu["cores"], "kind": "oracle",
            "sample": f"{cpu['rows']} of {wl.T} token rows ({cpu['experts']} expert MLPs), median of "
                      f"{cpu['steps']} runs of {cpu['sample_s']:.2f} s, scaled x{cpu['scale']:.0f} to a step",
        }
        ac = cpu.get("all_cores")
        if ac and "us_per_step" in ac:
            line["cpu_baseline_all_cores"] = {
                "value": round(ac["us_per_step"], 1), "unit": "us/step", "cores": ac["cores"], "kind": "oracle",
                "sample": f"all {wl.T} token rows of the step at once, one persistent spawned process per row "
                          f"(the oracle unchanged, one BLAS thread each), wall time, median of {ac['steps']}; "
                          f"rows equal the single-thread run's",
            }
        elif ac:
            line["cpu_baseline_all_cores"] = ac
    if also:
        line["also"] = also
    main["step"].close()
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args):
    """The oracle as the reference arm, on the host cores (rank 0 only): whole
    steps, every token row at once in its own process, so ms_per_step x steps
    is the wall time of the timed steps. A workload with more rows than host
    cores falls back to a single-thread sample of rows, scaled to a step."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import synth
    wl = synth.WORKLOADS[args.workload]
    if wl.T <= (os.cpu_count() or 1):
        r = oracle_all_cores(args.seed, wl.name, args.steps, None, args.warmup)
        v = round(r["us_mean"], 1)
        sample = (f"all {wl.T} token rows of every step at once, one spawned process per row (the oracle "
                  f"unchanged, one BLAS thread each); {args.warmup} untimed steps, then {args.steps} timed; "
                  f"value = mean wall time per step (median {r['us_per_step']:.0f} us)")
        cores = r["cores"]
    else:
        ctx = mp.get_context("spawn")
        q = ctx.Queue()
        p = ctx.Process(target=oracle_baseline, args=(args.seed, wl.name, args.steps, args.warmup, q, None, False))
        p.start()
        r = q.get(timeout=3600)
        p.join(timeout=60)
        v = round(r["us_per_step"], 1)
        sample = (f"{r['rows']} of {wl.T} token rows ({r['experts']} expert MLPs) per step on one thread, "
                  f"scaled x{r['scale']:.0f} to a step")
        cores = r["cores"]
    line = {
        "impl": "reference",
        "metric": "MoE step us & achieved HBM GB/s (% of roofline) at 6/24/96/384 token rows",
        "value": v, "unit": "us/step", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(v / 1e3, 3), "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 (oracle)", "data": "synthetic (seeded counter-based generator)",
        "config": bench_config(wl, args, world),
        "cpu_baseline": {"value": v, "unit": "us/step", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=["tiny", "bs1", "bs4", "bs16", "bs64", "bs1_fp4", "bs4_fp4", "bs64_fp4"])
    ap.add_argument("--path", default="auto", choices=list(PATH_FLAGS),
                    help="expert kernel: auto (the library default: mma), or pin gemv / mma")
    ap.add_argument("--fused", type=int, default=0, choices=[0, 1, 2, 3, 4],
                    help="time only the fused step (router projection + this many residual streams with "
                         "RMSNorm + MXFP8) on the workload; prints its own line")
    ap.add_argument("--seed", type=int, default=42, help="seed of every synthetic input (default 42)")
    ap.add_argument("--l2", default="inputs", choices=["inputs", "flush"],
                    help="between timed steps: no flush, the step's weights being larger than L2 (inputs), or an "
                         "L2 flush (flush); the other policy is reported beside the value")
    ap.add_argument("--clocks-log", default=None,
                    help="also write the raw nvidia-smi clock samples of the timed region to this CSV file")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-others", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--experts", type=int, default=0,
                    help="smaller expert count for profiling captures (default: the workload's E)")
    ap.add_argument("--layer-copies", type=int, default=LAYER_COPIES,
                    help=f"copies of the layer's weights the timed steps cycle through (default {LAYER_COPIES}; "
                         "1 keeps a profiling capture's device memory small)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    args.layer_copies = max(1, args.layer_copies)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
