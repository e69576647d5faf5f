"""Build libmambascan.so in-tree with nvcc for sm_103a (B300)."""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libmambascan.so")
# One translation unit per kernel family (each becomes its own device module), compiled in
# parallel and linked into one shared library.
SOURCES = ["mamba_scan.cu", "fwd_lane_f32.cu", "fwd_lane_bf16.cu", "fwd_warp_f32.cu", "fwd_warp_bf16.cu", "bwd.cu",
           "conv.cu", "step.cu", "fwd_plan.cu"]
HEADERS = ["host.cuh", "fwd_common.cuh", "fwd_lane.cuh", "fwd_warp.cuh", "ptx.cuh", "common.cuh", "scan_fwd.cuh", "scan_fwd_cl.cuh", "scan_fix.cuh",
           "scan_bwd.cuh", "state_step.cuh", "conv.cuh"]
OBJDIR = os.path.join(HERE, "_build")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC",
    "--expt-relaxed-constexpr",
]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return "nvcc"


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "mamba_scan.h")]
    return any(os.path.getmtime(p) > t for p in deps if os.path.exists(p))


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Compile when a source is newer than the library (or when forced).  cudart is linked
    statically (nvcc's default), so the library only needs the driver at run time."""
    if not force and not stale():
        return LIB
    os.makedirs(OBJDIR, exist_ok=True)
    inc = ["-I", os.path.join(ROOT, "include"), "-I", CSRC]

    def compile_one(src: str) -> str:
        obj = os.path.join(OBJDIR, os.path.splitext(src)[0] + f".{os.getpid()}.o")
        cmd = [_nvcc(), *NVCC_FLAGS, *extra, *inc, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.check_call(cmd)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as pool:
        objs = list(pool.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [_nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    for o in objs:
        os.remove(o)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True,
          extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else [])
