"""The golden fixture of the tiny fp32 scan workload (tests/golden/tiny_scan.json, written by
tests/golden/make_golden.py from the oracle only).

On the CPU it guards the oracle and the input recipe against silent change: the seeded generator
still produces the stored inputs bit for bit, and the oracle still produces the stored outputs.
On the GPU both forward kernels and the decode step are compared with the stored outputs under the
fp32 bound (max|y_gpu - y_ref| / max|y_ref| <= 1e-4), without running the oracle.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_scan.json")


def _load():
    with open(GOLDEN) as f:
        g = json.load(f)
    s = g["shape"]
    b, d, n, L = s["batch"], s["dim"], s["dstate"], s["seqlen"]
    shapes = {"u": (b, d, L), "delta": (b, d, L), "z": (b, d, L), "B": (b, n, L), "C": (b, n, L), "A": (d, n),
              "D": (d,), "delta_bias": (d,)}
    inp = {k: np.asarray(g["inputs"][k], np.float32).reshape(shp) for k, shp in shapes.items()}
    step = {k: np.asarray(v, np.float32).reshape((b, d) if k in ("x", "delta", "z") else (b, n))
            for k, v in g["step_inputs"].items()}
    out = {"y": np.asarray(g["y"]).reshape(b, d, L), "last_state": np.asarray(g["last_state"]).reshape(b, d, n),
           "step_y": np.asarray(g["step_y"]).reshape(b, d), "step_state": np.asarray(g["step_state"]).reshape(b, d, n)}
    return inp, step, out


def test_recipe_still_gives_the_stored_inputs():
    inp, _, _ = _load()
    now = synth.scan_inputs(synth.CONFIGS["tiny"])
    for k, v in inp.items():
        assert np.array_equal(np.asarray(now[k], np.float32), v), k


def test_oracle_still_gives_the_stored_outputs():
    inp, step, out = _load()
    y, st = oracle.scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["delta_bias"],
                        True, "f32", nthreads=1)
    assert np.array_equal(y, out["y"]) and np.array_equal(st, out["last_state"])
    state = np.array(st, dtype=np.float64)
    ys = oracle.state_step(state, step["x"], step["delta"], inp["A"], step["B"], step["C"], inp["D"], step["z"],
                           inp["delta_bias"], True, "f32")
    assert np.array_equal(ys, out["step_y"]) and np.array_equal(state, out["step_state"])


def _rel(got, ref):
    return float(np.max(np.abs(np.asarray(got, np.float64) - ref)) / max(np.max(np.abs(ref)), 1e-30))


@pytest.mark.gpu
@pytest.mark.parametrize("kernel", ["lane", "warp"])
def test_gpu_matches_the_stored_outputs(kernel):
    import torch
    import sequence_scan_selective_b300 as ms
    inp, step, out = _load()
    t = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in inp.items()}
    old = os.environ.get("MAMBA_SCAN_KERNEL")
    os.environ["MAMBA_SCAN_KERNEL"] = kernel
    try:
        y, st = ms.mamba_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True)
        torch.cuda.synchronize()
    finally:
        if old is None:
            os.environ.pop("MAMBA_SCAN_KERNEL", None)
        else:
            os.environ["MAMBA_SCAN_KERNEL"] = old
    assert _rel(y.cpu().numpy(), out["y"]) <= 1e-4
    assert _rel(st.cpu().numpy(), out["last_state"]) <= 1e-4
    s = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in step.items()}
    ys = ms.mamba_state_step(st, s["x"], s["delta"], t["A"], s["B"], s["C"], t["D"], s["z"], t["delta_bias"], True)
    torch.cuda.synchronize()
    assert _rel(ys.cpu().numpy(), out["step_y"]) <= 1e-4
    assert _rel(st.cpu().numpy(), out["step_state"]) <= 1e-4
