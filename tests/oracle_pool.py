"""The oracle's expert MLPs over many token rows, one expert per task, in a
pool of spawned processes (test infrastructure).

A full-size step touches up to 257 experts of 3 x 2048 x 4096 weights each.
Drawing and quantising one expert's weights on the host takes seconds, so the
parity tests at the benchmark's sizes hand the experts to worker processes.
Each task draws one expert's weights once and runs oracle.expert_mlp for every
batch of token rows that chose it. It also returns sum_k |x_k w_k| for the gate
and the up projection, which bound the device's fp32 accumulation error in
the h check. No arithmetic of the method is done here; every value comes from
the oracle's own functions.

The pool uses the spawn start method, so it can be started after CUDA is
initialised in the parent, and each worker runs BLAS on one thread.
"""
from __future__ import annotations

import os

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import multiprocessing as mp  # noqa: E402
from concurrent.futures import ProcessPoolExecutor  # noqa: E402

import numpy as np  # noqa: E402


WEIGHT_FIELDS = ("w_gate", "s_gate", "w_up", "s_up", "w_down", "s_down")


def sha256_of(a) -> str:
    import hashlib
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def expert_task(args):
    """args = (seed, e, H, I, fmt, swiglu_limit, jobs); jobs = [(tag, xq, xs), ...].
    Returns (e, {tag: (g, u, h, hq, hs, o, sum_g, sum_u)}, {field: sha256 of the
    oracle's quantised weight tensor})."""
    import oracle
    seed, e, H, I, fmt, lim, jobs = args
    w = oracle.expert_weights_from_synth(seed, e, H, I, fmt=fmt)
    hashes = {n: sha256_of(getattr(w, n)) for n in WEIGHT_FIELDS}
    ag = np.abs(w.dequant("gate"))
    au = np.abs(w.dequant("up"))
    out = {}
    for tag, xq, xs in jobs:
        g, u, h, hq, hs, o = oracle.expert_mlp(xq, xs, w, lim)
        ax = np.abs(oracle.mxfp8_dequantize(xq, xs))
        out[tag] = (g, u, h, hq, hs, o, ax @ ag.T, ax @ au.T)
    return e, out, hashes


def run_experts(tasks, workers=None):
    """Runs expert_task over `tasks` in a spawn pool; returns
    ({e: {tag: result}}, {e: weight hashes}). The tasks with the most token
    rows start first. A worker that dies raises (BrokenProcessPool) instead of
    being replaced, so a failing pool ends the test rather than stalling it."""
    n = workers or max(1, min(len(tasks), os.cpu_count() or 1, 32))
    order = sorted(tasks, key=lambda t: -sum(len(j[1]) for j in t[6]))
    res, hashes = {}, {}
    with ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn")) as ex:
        for e, out, h in ex.map(expert_task, order):
            res[e], hashes[e] = out, h
    return res, hashes
