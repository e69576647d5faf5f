"""GPU parity of the recurrent decode step (in-place state update) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, dev_inputs, from_dev, rel_err, sample_rows, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ms():
    import sequence_scan_selective_b300 as m
    return m


def _params_dev(p):
    return {k: torch.from_numpy(np.ascontiguousarray(v, np.float32)).cuda() for k, v in p.items()}


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 4, 5, 16, 24, 64])
def test_steps_match_oracle(ms, dtype, N):
    cfg = synth.CONFIGS["decode"].replace(batch=3, dim=50, dstate=N, dtype=dtype, decode_steps=20, seed=30 + N)
    p = synth.params(cfg)
    pd = _params_dev(p)
    h0 = synth.decode_state0(cfg)
    st_dev = torch.from_numpy(h0.copy()).cuda()
    st_ref = h0.astype(np.float64).copy()
    for s in range(cfg.decode_steps):
        inp = synth.decode_step_inputs(cfg, s)
        dv = {k: to_dev(v, dtype) for k, v in inp.items()}
        y = ms.mamba_state_step(st_dev, dv["x"], dv["delta"], pd["A"], dv["B"], dv["C"], pd["D"], dv["z"],
                                pd["delta_bias"], True)
        y_ref = oracle.state_step(st_ref, inp["x"], inp["delta"], p["A"], inp["B"], inp["C"], p["D"], inp["z"],
                                  p["delta_bias"], True, dtype)
        assert rel_err(from_dev(y), y_ref) <= TOL[dtype], f"step {s}"
    assert rel_err(from_dev(st_dev), st_ref) <= TOL[dtype]
    ms.device_status()


def test_delta_zero_keeps_state_bit_for_bit(ms):
    cfg = synth.CONFIGS["decode"].replace(batch=4, dim=96, decode_steps=1, dtype="f32")
    pd = _params_dev(synth.params(cfg))
    st = torch.from_numpy(synth.decode_state0(cfg)).cuda()
    before = st.clone()
    dv = {k: to_dev(v, "f32") for k, v in synth.decode_step_inputs(cfg, 0).items()}
    ms.mamba_state_step(st, dv["x"], torch.zeros_like(dv["delta"]), pd["A"], dv["B"], dv["C"], pd["D"], dv["z"],
                        None, False)
    torch.cuda.synchronize()
    assert torch.equal(st, before)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_scan_equals_successive_steps(ms, dtype):
    """The scan and L recurrent steps from a zero state describe the same recurrence (guide 2.4)."""
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=40, seqlen=48, dtype=dtype, seed=31)
    d = dev_inputs(synth.scan_inputs(cfg), dtype)
    y, last = ms.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"], True)
    st = torch.zeros((cfg.batch, cfg.dim, cfg.dstate), device="cuda")
    ys = []
    for t in range(cfg.seqlen):
        col = lambda k: d[k][:, :, t].contiguous()
        ys.append(ms.mamba_state_step(st, col("u"), col("delta"), d["A"], col("B"), col("C"), d["D"], col("z"),
                                      d["delta_bias"], True))
    ys = torch.stack(ys, dim=2)
    tol = 1e-5 if dtype == "f32" else 1e-2
    assert rel_err(from_dev(ys), from_dev(y)) <= tol
    assert rel_err(from_dev(st), from_dev(last)) <= 1e-5


def test_state_handoff_scan_then_decode(ms):
    """Prefill with the scan, continue with decode steps from its last_state."""
    cfg = synth.CONFIGS["b14"].replace(batch=2, dim=64, seqlen=130, seed=32)
    inp = synth.scan_inputs(cfg)
    d = dev_inputs(inp, cfg.dtype)
    pre = lambda k: d[k][:, :, :128].contiguous()
    _, last = ms.mamba_scan_fwd(pre("u"), pre("delta"), d["A"], pre("B"), pre("C"), d["D"], pre("z"),
                                d["delta_bias"], True)
    ys = []
    for t in (128, 129):
        col = lambda k: d[k][:, :, t].contiguous()
        ys.append(ms.mamba_state_step(last, col("u"), col("delta"), d["A"], col("B"), col("C"), d["D"], col("z"),
                                      d["delta_bias"], True))
    y_ref, st_ref = oracle.scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                inp["delta_bias"], True, cfg.dtype)
    assert rel_err(from_dev(torch.stack(ys, 2)), y_ref[:, :, 128:]) <= TOL["bf16"]
    assert rel_err(from_dev(last), st_ref) <= TOL["bf16"]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_workload_full_size(ms, dtype):
    """128 x 5120 x 16, fp32 state, 1000 successive steps with bf16 inputs (the primary reading of
    the decode workload) and with fp32 inputs; sampled channels vs oracle."""
    cfg = synth.CONFIGS["decode"].replace(dtype=dtype)
    p = synth.params(cfg)
    pd = _params_dev(p)
    allin = synth.decode_inputs(cfg)
    dev = {k: to_dev(v, cfg.dtype) for k, v in allin.items()}
    h0 = synth.decode_state0(cfg)
    st = torch.from_numpy(h0).cuda()
    ys = torch.empty((cfg.decode_steps, cfg.batch, cfg.dim), device="cuda",
                     dtype=torch.bfloat16 if dtype == "bf16" else torch.float32)
    for s in range(cfg.decode_steps):
        ms.mamba_state_step(st, dev["x"][s], dev["delta"][s], pd["A"], dev["B"][s], dev["C"][s], pd["D"],
                            dev["z"][s], pd["delta_bias"], True, y=ys[s])
    torch.cuda.synchronize()
    rows = sample_rows(cfg.batch * cfg.dim, 256, seed=3)
    rb, rd = rows // cfg.dim, rows % cfg.dim
    st_ref = h0.reshape(-1, cfg.dstate)[rows].astype(np.float64).copy()
    y_ref = np.empty((cfg.decode_steps, len(rows)))
    for s in range(cfg.decode_steps):
        y_ref[s] = oracle.state_step_rows(rows, cfg.dim, st_ref, allin["x"][s, rb, rd], allin["delta"][s, rb, rd],
                                          allin["z"][s, rb, rd], p["A"], p["D"], p["delta_bias"], allin["B"][s],
                                          allin["C"][s], True, cfg.dtype)
    idx = torch.from_numpy(rows).cuda()
    yg = from_dev(ys.reshape(cfg.decode_steps, -1)[:, idx])
    sg = from_dev(st.reshape(-1, cfg.dstate)[idx])
    assert rel_err(yg, y_ref) <= TOL[cfg.dtype]
    assert rel_err(sg, st_ref) <= TOL[cfg.dtype]
    del dev, st, ys
    torch.cuda.empty_cache()
