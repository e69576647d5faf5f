"""Writes the golden fixtures of this folder from the fp64 oracle (and nothing else).

tiny_scan.json: the tiny fp32 scan workload (batch 1, d_inner 16, N 4, L 64; A[d, n] = -(n+1);
Delta log-uniform in [1e-3, 0.1] through softplus with zero bias; u, z, B, C ~ N(0, 1); D = 1;
seed 0), its inputs as stored (fp32), the oracle's y and final state (fp64), and one decode step
from that final state with fresh inputs (the recurrent form: visual guide to Mamba and SSMs,
section 2.4).  Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402


def _f32(a):
    # 9 significant digits identify an fp32 value exactly
    return [float("%.9g" % v) for v in np.asarray(a, np.float32).ravel()]


def _f64(a):
    return [float(v) for v in np.asarray(a, np.float64).ravel()]


def main():
    cfg = synth.CONFIGS["tiny"]
    inp = synth.scan_inputs(cfg)
    y, st = oracle.scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["delta_bias"],
                        True, "f32", nthreads=1)
    rng = np.random.default_rng(12345)
    bsz, dim, N = cfg.batch, cfg.dim, cfg.dstate
    step = {"x": rng.standard_normal((bsz, dim)).astype(np.float32),
            "delta": rng.uniform(-4.0, -1.0, (bsz, dim)).astype(np.float32),
            "z": rng.standard_normal((bsz, dim)).astype(np.float32),
            "B": rng.standard_normal((bsz, N)).astype(np.float32),
            "C": rng.standard_normal((bsz, N)).astype(np.float32)}
    state = np.array(st, dtype=np.float64)
    y_step = oracle.state_step(state, step["x"], step["delta"], inp["A"], step["B"], step["C"], inp["D"], step["z"],
                               inp["delta_bias"], True, "f32")
    out = {
        "about": ("tiny fp32 scan workload (batch 1, d_inner 16, N 4, L 64; seed 0): inputs as stored, the fp64 "
                  "oracle's y and final state, then one decode step from that state; written by "
                  "tests/golden/make_golden.py from oracle/ only"),
        "shape": {"batch": bsz, "dim": dim, "dstate": N, "seqlen": cfg.seqlen},
        "inputs": {k: _f32(inp[k]) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias")},
        "y": _f64(y), "last_state": _f64(st),
        "step_inputs": {k: _f32(v) for k, v in step.items()},
        "step_y": _f64(y_step), "step_state": _f64(state),
    }
    with open(os.path.join(HERE, "tiny_scan.json"), "w") as f:
        json.dump(out, f, separators=(",", ":"))
        f.write("\n")


if __name__ == "__main__":
    main()
