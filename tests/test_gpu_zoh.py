"""GPU parity of the exact zero-order-hold discretisation (Bbar = (exp(Delta A) - 1) / A * B) in the
forward scan, the decode step and the backward pass, against the fp64 oracle's hold.

The workload recipe gives |Delta A| from 1e-3 to 1.6, so both of the kernels' evaluation branches
of the hold factor (Taylor series below |Delta A| = 1/4, closed form above) are exercised; one
case also sets A = 0 for a state.  Tolerances as for the simplified discretisation: 1e-4 (fp32
storage) and 2e-2 (bf16 storage), max-abs error over max-abs value per tensor.
"""
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


def _fwd(ms, inp, dtype, h0=None):
    d = dev_inputs(inp, dtype)
    h0t = None if h0 is None else torch.from_numpy(np.ascontiguousarray(h0, np.float32)).cuda()
    y, st = ms.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d.get("D"), d.get("z"),
                              d.get("delta_bias"), True, h0=h0t, disc="zoh")
    torch.cuda.synchronize()
    ms.device_status()
    return from_dev(y), from_dev(st)


def _check_fwd(ms, cfg, zero_state=False, h0=None):
    inp = synth.scan_inputs(cfg)
    if zero_state:
        inp["A"][:, 0] = 0.0
    y, st = _fwd(ms, inp, cfg.dtype, h0)
    y_ref, st_ref = oracle.scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                inp["delta_bias"], True, cfg.dtype, h0=h0, disc="zoh")
    ey, es = rel_err(y, y_ref), rel_err(st, st_ref)
    assert ey <= TOL[cfg.dtype] and es <= TOL[cfg.dtype], (ey, es)
    # and the hold is really in effect: the simplified discretisation differs by more than the bound
    if cfg.dtype == "f32":
        y_simple, _ = oracle.scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                  inp["delta_bias"], True, cfg.dtype, h0=h0)
        assert rel_err(y, y_simple) > 3 * TOL[cfg.dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("L", [1, 33, 200, 1000])
def test_zoh_fwd_ragged(ms, dtype, L):
    _check_fwd(ms, synth.CONFIGS["m130"].replace(batch=2, dim=40, seqlen=L, dtype=dtype, seed=300 + L))


@pytest.mark.parametrize("N", [4, 16, 32, 64])
def test_zoh_fwd_state_sizes(ms, N):
    _check_fwd(ms, synth.CONFIGS["m130"].replace(batch=2, dim=24, dstate=N, seqlen=160, seed=310 + N),
               zero_state=True)


def test_zoh_fwd_split_sequence_with_initial_state(ms):
    """Few channels and a long sequence: the time axis is split into segments (carry pass)."""
    cfg = synth.CONFIGS["long"].replace(dim=16, seqlen=20000, seed=320)
    h0 = np.random.default_rng(321).standard_normal((1, 16, 16)).astype(np.float32)
    _check_fwd(ms, cfg, h0=h0)


def test_zoh_fwd_full_size_sampled(ms):
    cfg = synth.CONFIGS["m130"]
    inp = synth.scan_inputs(cfg)
    y, st = _fwd(ms, inp, cfg.dtype)
    rows = sample_rows(cfg.batch * cfg.dim, 24, seed=5)
    r = lambda a, w: a.reshape(cfg.batch * cfg.dim, w)[rows]
    y_ref, st_ref = oracle.scan_rows(rows, cfg.dim, r(inp["u"], cfg.seqlen), r(inp["delta"], cfg.seqlen),
                                     r(inp["z"], cfg.seqlen), inp["A"], inp["D"], inp["delta_bias"], inp["B"],
                                     inp["C"], True, cfg.dtype, disc="zoh")
    assert rel_err(r(y, cfg.seqlen), y_ref) <= TOL[cfg.dtype]
    assert rel_err(r(st, cfg.dstate), st_ref) <= TOL[cfg.dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zoh_decode_steps(ms, dtype):
    cfg = synth.CONFIGS["decode"].replace(batch=4, dim=96, dtype=dtype, seed=330)
    p = synth.params(cfg)
    p["A"][:, 3] = 0.0
    state0 = synth.decode_state0(cfg)
    st_gpu = torch.from_numpy(state0.copy()).cuda()
    st_ref = state0.astype(np.float64).copy()
    A = torch.from_numpy(p["A"]).cuda()
    D = torch.from_numpy(p["D"]).cuda()
    bias = torch.from_numpy(p["delta_bias"]).cuda()
    for step in range(12):
        s = synth.decode_step_inputs(cfg, step)
        y = ms.mamba_state_step(st_gpu, to_dev(s["x"], dtype), to_dev(s["delta"], dtype), A,
                                to_dev(s["B"], dtype), to_dev(s["C"], dtype), D, to_dev(s["z"], dtype), bias,
                                True, disc="zoh")
        y_ref = oracle.state_step(st_ref, s["x"], s["delta"], p["A"], s["B"], s["C"], p["D"], s["z"],
                                  p["delta_bias"], True, dtype, disc="zoh")
        torch.cuda.synchronize()
        assert rel_err(from_dev(y), y_ref) <= TOL[dtype], step
    assert rel_err(from_dev(st_gpu), st_ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype,L,N", [("f32", 77, 16), ("bf16", 200, 16), ("f32", 1000, 5), ("f32", 2048, 16)])
def test_zoh_bwd(ms, dtype, L, N):
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=72, dstate=N, seqlen=L, dtype=dtype, seed=340 + L)
    inp = synth.scan_inputs(cfg)
    inp["A"][:, 0] = 0.0
    g = synth.grad_inputs(cfg)
    d = dev_inputs(inp, dtype)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    out = ms.mamba_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], to_dev(g["dy"], dtype), d["D"], d["z"],
                            d["delta_bias"], True, h0=f32(g["h0"]), dlast_state=f32(g["dlast"]), disc="zoh")
    torch.cuda.synchronize()
    ref = oracle.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], synth.widen(g["dy"], dtype),
                          inp["D"], inp["z"], inp["delta_bias"], True, dtype, h0=g["h0"], dlast_state=g["dlast"],
                          disc="zoh")
    errs = {k: rel_err(from_dev(out[k]), ref[k]) for k in ref if ref[k] is not None}
    bad = {k: v for k, v in errs.items() if not v <= TOL[dtype]}
    assert not bad, (bad, errs)
