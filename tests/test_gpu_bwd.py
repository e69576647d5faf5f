"""GPU parity of the backward pass (gradients with recomputed states) against the fp64 oracle.

Every gradient is compared as max|g_gpu - g_oracle| / max|g_oracle| per tensor, with the forward
scan's bounds: 1e-4 with fp32 storage, 2e-2 with bf16 storage (du, ddelta, dz are stored in the
input dtype; dA, dB, dC, dD, ddelta_bias and dh0 are fp32).  Both sides see the same stored
inputs (bf16 values widened exactly).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, dev_inputs, from_dev, rel_err, sample_rows, to_dev

pytestmark = pytest.mark.gpu

GRADS = ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0")


@pytest.fixture(scope="module")
def ms():
    import sequence_scan_selective_b300 as m
    return m


def _inputs(cfg, drop=(), with_h0=True, with_dlast=True):
    inp = synth.scan_inputs(cfg)
    g = synth.grad_inputs(cfg)
    inp["dy"] = g["dy"]
    inp["h0"] = g["h0"] if with_h0 else None
    inp["dlast"] = g["dlast"] if with_dlast else None
    for k in drop:
        inp[k] = None
    return inp


def _gpu(ms, inp, dtype, softplus=True):
    d = dev_inputs(inp, dtype)
    dy = to_dev(inp["dy"], dtype)
    f32 = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    out = ms.mamba_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], dy, d.get("D"), d.get("z"),
                            d.get("delta_bias"), softplus, h0=f32(inp["h0"]), dlast_state=f32(inp["dlast"]))
    torch.cuda.synchronize()
    return {k: (None if v is None else from_dev(v)) for k, v in out.items()}


def _oracle(inp, dtype, softplus=True):
    return oracle.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"],
                           synth.widen(inp["dy"], dtype), inp.get("D"), inp.get("z"), inp.get("delta_bias"),
                           softplus, dtype, h0=inp["h0"], dlast_state=inp["dlast"])


def _compare(got, ref, dtype, names=GRADS):
    errs = {}
    for k in names:
        if ref.get(k) is None or got.get(k) is None:
            continue
        errs[k] = rel_err(got[k], ref[k])
    bad = {k: v for k, v in errs.items() if not v <= TOL[dtype]}
    assert not bad, f"gradients off: {bad} (all: {errs})"
    return errs


def _check(ms, cfg, softplus=True, **kw):
    inp = _inputs(cfg, **kw)
    got = _gpu(ms, inp, cfg.dtype, softplus)
    ref = _oracle(inp, cfg.dtype, softplus)
    if inp["h0"] is None:
        ref["dh0"] = None
    return _compare(got, ref, cfg.dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("L", [1, 7, 16, 17, 32, 77, 200, 1000])
def test_bwd_ragged_lengths(ms, dtype, L):
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=40, seqlen=L, dtype=dtype, seed=100 + L)
    _check(ms, cfg)


@pytest.mark.parametrize("N", [1, 4, 5, 13, 16])
def test_bwd_state_sizes(ms, N):
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=33, dstate=N, seqlen=96, seed=120 + N)
    _check(ms, cfg)


@pytest.mark.parametrize("drop,softplus,h0,dlast", [
    (("z",), True, True, True),
    (("D", "delta_bias"), True, False, False),
    ((), False, False, True),
    (("z", "D", "delta_bias"), False, True, False),
])
def test_bwd_optional_inputs(ms, drop, softplus, h0, dlast):
    cfg = synth.CONFIGS["m130"].replace(batch=3, dim=64, seqlen=128, seed=140 + len(drop))
    inp = _inputs(cfg, drop=drop, with_h0=h0, with_dlast=dlast)
    if not softplus:  # Delta = delta + bias must stay positive: place it in (0, 0.1]
        step = np.abs(inp["delta"]).astype(np.float32) * np.float32(0.02)
        bias = inp["delta_bias"] if inp["delta_bias"] is not None else np.zeros(cfg.dim, np.float32)
        inp["delta"] = (step - bias[None, :, None]).astype(np.float32)
    got = _gpu(ms, inp, cfg.dtype, softplus)
    ref = _oracle(inp, cfg.dtype, softplus)
    for k in ("dz", "dD", "ddelta_bias", "dh0"):
        want_none = {"dz": "z", "dD": "D", "ddelta_bias": "delta_bias"}.get(k)
        if (want_none and inp.get(want_none) is None) or (k == "dh0" and inp["h0"] is None):
            assert got[k] is None
            ref[k] = None
    _compare(got, ref, cfg.dtype)


def test_bwd_medium_shape(ms):
    """Several CTAs per batch row, many tiles, both sweeps long."""
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=256, seqlen=2048, seed=150)
    _check(ms, cfg)


@pytest.mark.parametrize("name", ["m130", "b14"])
def test_bwd_full_size_sampled(ms, name):
    """The full workload on the GPU; the oracle checks sampled channels (their per-channel
    gradients), all batch rows of sampled channels (dA, dD, ddelta_bias) and every channel of
    batch row 0 (dB, dC of that row)."""
    cfg = synth.CONFIGS[name]
    inp = _inputs(cfg)
    got = _gpu(ms, inp, cfg.dtype)
    bsz, dim, L, N = cfg.batch, cfg.dim, cfg.seqlen, cfg.dstate
    r = lambda a, w: a.reshape(bsz * dim, w)
    chans = np.unique(sample_rows(dim, 6, seed=7))
    rows = np.array(sorted({b * dim + int(d) for b in range(bsz) for d in chans}), dtype=np.int64)
    z = r(inp["z"], L)[rows]
    ref = oracle.scan_bwd_rows(rows, bsz, dim, r(inp["u"], L)[rows], r(inp["delta"], L)[rows], z,
                               inp["A"], inp["D"], inp["delta_bias"], inp["B"], inp["C"],
                               synth.widen(r(inp["dy"], L)[rows], cfg.dtype), True, cfg.dtype,
                               r(inp["h0"], N)[rows], r(inp["dlast"], N)[rows])
    errs = {}
    for k in ("du", "ddelta", "dz"):
        errs[k] = rel_err(r(got[k], L)[rows], ref[k])
    errs["dh0"] = rel_err(r(got["dh0"], N)[rows], ref["dh0"])
    for k in ("dA",):
        errs[k] = rel_err(got[k][chans], ref[k][chans])
    for k in ("dD", "ddelta_bias"):
        errs[k] = rel_err(got[k][chans], ref[k][chans])
    row0 = np.arange(dim)
    ref0 = oracle.scan_bwd_rows(row0, bsz, dim, r(inp["u"], L)[row0], r(inp["delta"], L)[row0],
                                r(inp["z"], L)[row0], inp["A"], inp["D"], inp["delta_bias"], inp["B"],
                                inp["C"], synth.widen(r(inp["dy"], L)[row0], cfg.dtype), True, cfg.dtype,
                                r(inp["h0"], N)[row0], r(inp["dlast"], N)[row0])
    errs["dB"] = rel_err(got["dB"][0], ref0["dB"][0])
    errs["dC"] = rel_err(got["dC"][0], ref0["dC"][0])
    bad = {k: v for k, v in errs.items() if not v <= TOL[cfg.dtype]}
    assert not bad, f"{name}: {bad} (all: {errs})"


def test_bwd_empty_sequence(ms):
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=8, dstate=4, seqlen=0, seed=160)
    dl = torch.randn((2, 8, 4), device="cuda")
    h0 = torch.randn((2, 8, 4), device="cuda")
    e = torch.zeros((2, 8, 0), device="cuda")
    be = torch.zeros((2, 4, 0), device="cuda")
    A = -torch.ones((8, 4), device="cuda")
    out = ms.mamba_scan_bwd(e, e, A, be, be, e, torch.ones(8, device="cuda"), None, None, True, h0=h0,
                            dlast_state=dl)
    torch.cuda.synchronize()
    assert torch.equal(out["dh0"], dl)
    assert torch.count_nonzero(out["dA"]) == 0 and torch.count_nonzero(out["dD"]) == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [17, 24, 32, 48, 64])
def test_bwd_wide_state(ms, dtype, N):
    """N > 16 runs one launch per block of 16 states; the per-(channel, step) gradients, which sum
    over all states, are accumulated across the launches in fp32."""
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=33, dstate=N, seqlen=150, dtype=dtype, seed=180 + N)
    _check(ms, cfg)


@pytest.mark.parametrize("disc", ["simple", "zoh"])
def test_bwd_wide_state_optional_inputs(ms, disc):
    cfg = synth.CONFIGS["m130"].replace(batch=1, dim=40, dstate=40, seqlen=77, seed=190)
    inp = _inputs(cfg, drop=("z", "D"))
    d = dev_inputs(inp, cfg.dtype)
    f32 = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    got = ms.mamba_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], to_dev(inp["dy"], cfg.dtype), None, None,
                            d.get("delta_bias"), True, h0=f32(inp["h0"]), dlast_state=f32(inp["dlast"]), disc=disc)
    torch.cuda.synchronize()
    got = {k: (None if v is None else from_dev(v)) for k, v in got.items()}
    ref = oracle.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], synth.widen(inp["dy"], cfg.dtype),
                          None, None, inp.get("delta_bias"), True, cfg.dtype, h0=inp["h0"],
                          dlast_state=inp["dlast"], disc=disc)
    _compare(got, ref, cfg.dtype)


class _env:
    def __init__(self, **kv):
        self.kv, self.old = kv, {}

    def __enter__(self):
        import os
        for k, v in self.kv.items():
            self.old[k] = os.environ.get(k)
            os.environ[k] = v

    def __exit__(self, *exc):
        import os
        for k, v in self.old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("nseg", [2, 5])
def test_bwd_split_time_axis(ms, dtype, nseg):
    """The time axis split into segments (carry launch, full launch per segment, correction
    launch from each segment's end) gives the oracle's gradients."""
    cfg = synth.CONFIGS["long"].replace(batch=2, dim=40, seqlen=6000, dtype=dtype, seed=200 + nseg)
    with _env(MAMBA_SCAN_BWD_NSEG=str(nseg)):
        _check(ms, cfg)


@pytest.mark.parametrize("disc", ["simple", "zoh"])
def test_bwd_split_options(ms, disc):
    """Split time axis with the hold, without z and D, and with 24 states (two state blocks)."""
    cfg = synth.CONFIGS["long"].replace(batch=1, dim=33, dstate=24, seqlen=3001, seed=210)
    inp = _inputs(cfg, drop=("z", "D"))
    d = dev_inputs(inp, cfg.dtype)
    f32 = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    with _env(MAMBA_SCAN_BWD_NSEG="4"):
        got = ms.mamba_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], to_dev(inp["dy"], cfg.dtype), None,
                                None, d.get("delta_bias"), True, h0=f32(inp["h0"]), dlast_state=f32(inp["dlast"]),
                                disc=disc)
        torch.cuda.synchronize()
    got = {k: (None if v is None else from_dev(v)) for k, v in got.items()}
    ref = oracle.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], synth.widen(inp["dy"], cfg.dtype),
                          None, None, inp.get("delta_bias"), True, cfg.dtype, h0=inp["h0"],
                          dlast_state=inp["dlast"], disc=disc)
    _compare(got, ref, cfg.dtype)


def test_bwd_split_without_decay(ms):
    """States with A = 0 never forget: the gradient carried into a segment reaches all of it, so
    the correction launch walks the whole segment."""
    cfg = synth.CONFIGS["long"].replace(batch=1, dim=24, seqlen=4000, seed=220)
    inp = _inputs(cfg)
    inp["A"] = inp["A"].copy()
    inp["A"][:, :2] = 0.0
    inp["A"][3, :] = 0.0
    got = None
    with _env(MAMBA_SCAN_BWD_NSEG="3"):
        got = _gpu(ms, inp, cfg.dtype)
    ref = _oracle(inp, cfg.dtype)
    _compare(got, ref, cfg.dtype)


def test_bwd_segment_count_invariance(ms):
    cfg = synth.CONFIGS["long"].replace(batch=1, dim=32, seqlen=8192, seed=230)
    inp = _inputs(cfg)
    outs = []
    for nseg in ("1", "4", "16"):
        with _env(MAMBA_SCAN_BWD_NSEG=nseg):
            outs.append(_gpu(ms, inp, cfg.dtype))
    for o in outs[1:]:
        for k in GRADS:
            if o.get(k) is not None:
                assert rel_err(o[k], outs[0][k]) <= 1e-5, k


def test_bwd_rejects_unsupported(ms):
    cfg = synth.CONFIGS["m130"].replace(batch=1, dim=8, dstate=16, seqlen=16, seed=170)
    inp = _inputs(cfg)
    d = dev_inputs(inp, "f32")
    with pytest.raises(ms.MambaScanError):  # a gradient output that aliases an input
        ms.mamba_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], to_dev(inp["dy"], "f32"), d["D"],
                          d["z"], d["delta_bias"], out={"du": d["u"], "ddelta": torch.empty_like(d["u"]),
                                                        "dz": None, "dA": torch.empty_like(d["A"]),
                                                        "dB": torch.empty_like(d["B"]),
                                                        "dC": torch.empty_like(d["C"]), "dD": None,
                                                        "ddelta_bias": None, "dh0": None})


def test_bwd_million_steps_library_plan(ms):
    """2^20 steps on few channels, with the library's own split of the time axis (no forced
    count: here 128 segments on a 148-SM device), against the oracle's gradients of every tensor."""
    cfg = synth.CONFIGS["long"].replace(batch=1, dim=64, seed=240)
    inp = _inputs(cfg)
    n0 = ms.launch_count()
    got = _gpu(ms, inp, cfg.dtype)
    assert ms.launch_count() - n0 >= 3  # carry, full and correction launches
    ref = _oracle(inp, cfg.dtype)
    _compare(got, ref, cfg.dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("nseg,N", [("1", 16), ("3", 16), ("1", 24)])
def test_bwd_register_budgets_agree(ms, dtype, nseg, N):
    """The 3-CTA-per-SM build of the backward kernel (which keeps each step's Abar from the slot's
    recomputation) gives the 4-CTA build's gradients, unsplit and split, one and two state
    blocks, and both match the oracle.  The per-(channel, step) gradients and dh0 come from one
    lane each and agree bit for bit; dA, dB, dC, dD and the bias gradient are sums that CTAs add
    into with atomics, whose order varies from run to run, so they agree to rounding."""
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=72, dstate=N, seqlen=1600, dtype=dtype, seed=230 + N)
    inp = _inputs(cfg)
    got = {}
    for minb in ("3", "4"):
        with _env(MAMBA_SCAN_BWD_MINB=minb, MAMBA_SCAN_BWD_NSEG=nseg):
            got[minb] = _gpu(ms, inp, dtype)
    for k in ("du", "ddelta", "dz", "dh0"):
        assert np.array_equal(got["3"][k], got["4"][k]), k
    for k in ("dA", "dB", "dC", "dD", "ddelta_bias"):
        assert rel_err(got["3"][k], got["4"][k]) <= 1e-5, k
    _compare(got["3"], _oracle(inp, dtype), dtype)
