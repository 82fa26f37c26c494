"""In-tree build of the CUDA libraries for sm_103a.

``build()`` compiles:
* ``csrc/*.cu`` -> ``moe_expert_layer_top_gb300/_build/libmoe.so``, the C-ABI library;
* the same sources with ``-DMOE_DEBUG_BOUNDS`` -> ``_build/libmoe_debug.so``, the
  bounds-checked build (every kernel index checked; a miss is reported as
  MOE_ERR_DEVICE_BOUNDS and the access skipped), loaded instead of libmoe.so
  when the environment sets MOE_DEBUG_BOUNDS=1;
* ``synth/synth.cu`` -> ``synth/_build/libmoe_synth.so``, the device side of the
  seeded input generator.
The translation units are compiled in parallel, each with one ``-gencode``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(LIB_DIR, "libmoe.so")
DEBUG_DIR = os.path.join(LIB_DIR, "debug")
DEBUG_LIB_PATH = os.path.join(LIB_DIR, "libmoe_debug.so")
SYNTH_DIR = os.path.join(ROOT, "synth")
SYNTH_LIB_DIR = os.path.join(SYNTH_DIR, "_build")
SYNTH_LIB_PATH = os.path.join(SYNTH_LIB_DIR, "libmoe_synth.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed: " + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def _compile(src: str, obj: str, extra=()):
    return _run([nvcc(), *ARCH, *FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj])


def _stale(target: str, sources) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(LIB_DIR, exist_ok=True)
    os.makedirs(DEBUG_DIR, exist_ok=True)
    os.makedirs(SYNTH_LIB_DIR, exist_ok=True)
    cus = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))
    deps = cus + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    deps.append(os.path.join(INCLUDE, "moe.h"))
    synth_src = os.path.join(SYNTH_DIR, "synth.cu")
    jobs = []
    if force or _stale(LIB_PATH, deps):
        objs = [os.path.join(LIB_DIR, os.path.basename(c)[:-3] + ".o") for c in cus]
        jobs.append(("moe", cus, objs, LIB_PATH, ()))
    if force or _stale(DEBUG_LIB_PATH, deps):
        objs = [os.path.join(DEBUG_DIR, os.path.basename(c)[:-3] + ".o") for c in cus]
        jobs.append(("moe_debug", cus, objs, DEBUG_LIB_PATH, ("-DMOE_DEBUG_BOUNDS",)))
    if force or _stale(SYNTH_LIB_PATH, [synth_src]):
        jobs.append(("synth", [synth_src], [os.path.join(SYNTH_LIB_DIR, "synth.o")], SYNTH_LIB_PATH, ()))
    work = [(s, o, tuple(flags) + (("-Xptxas", "-v") if verbose else ()))
            for _, srcs, objs, _, flags in jobs for s, o in zip(srcs, objs)]
    with ThreadPoolExecutor(max_workers=max(1, min(len(work), os.cpu_count() or 4))) as ex:
        logs = list(ex.map(lambda a: _compile(*a), work))
    if verbose:
        for log in logs:
            print(log)
    for _, _, objs, lib, _ in jobs:
        tmp = lib + ".tmp"
        _run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, lib)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
