"""GPU parity of the scan with the block's causal depthwise convolution fused in front of it
(mamba_scan_fwd_conv) against the fp64 oracle: the oracle's convolution gives u in fp64 and the
oracle's scan consumes it as it is (every other input widened exactly to fp64).  Tolerances as for
the scan: 1e-4 (fp32 storage), 2e-2 (bf16 storage).
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


def _f64(a, dtype):
    return synth.widen(a, dtype)


def _oracle(inp, cp, dtype, silu, prev=None, h0=None, disc="simple", rows=None):
    """Oracle of the fused call, for all channels or the flat channel rows ``rows``."""
    bsz, dim, L = inp["u"].shape
    r = lambda a, w: a.reshape(bsz * dim, w)
    rows = np.arange(bsz * dim) if rows is None else rows
    K = cp["conv_w"].shape[1]
    u = oracle.causal_conv_rows(rows, dim, r(inp["u"], L)[rows], cp["conv_w"], cp["conv_bias"], silu, dtype,
                                None if prev is None else r(prev, K - 1)[rows].astype(np.float64))
    return oracle.scan_rows(rows, dim, u, _f64(r(inp["delta"], L)[rows], dtype),
                            _f64(r(inp["z"], L)[rows], dtype), inp["A"], inp["D"], inp["delta_bias"],
                            _f64(inp["B"], dtype), _f64(inp["C"], dtype), True, "f64",
                            None if h0 is None else r(h0, inp["A"].shape[1])[rows].astype(np.float64), disc=disc)


def _gpu(ms, inp, cp, dtype, silu, prev=None, h0=None, disc="simple"):
    d = dev_inputs(inp, dtype)
    f = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    y, st = ms.mamba_scan_fwd_conv(d["u"], f(cp["conv_w"]), f(cp["conv_bias"]), d["delta"], d["A"], d["B"], d["C"],
                                   d["D"], d["z"], d["delta_bias"], True, conv_silu=silu, conv_prev=f(prev),
                                   h0=f(h0), disc=disc)
    torch.cuda.synchronize()
    ms.device_status()
    return from_dev(y), from_dev(st)


def _check(ms, cfg, K=4, silu=True, with_prev=False, disc="simple"):
    inp = synth.scan_inputs(cfg)
    cp = synth.conv_params(cfg, K)
    prev = synth.conv_prev(cfg, K) if with_prev else None
    y, st = _gpu(ms, inp, cp, cfg.dtype, silu, prev, disc=disc)
    y_ref, st_ref = _oracle(inp, cp, cfg.dtype, silu, prev, disc=disc)
    bsz, dim, L = inp["u"].shape
    ey = rel_err(y.reshape(bsz * dim, L), y_ref)
    es = rel_err(st.reshape(bsz * dim, -1), st_ref)
    assert ey <= TOL[cfg.dtype] and es <= TOL[cfg.dtype], (ey, es)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("L", [1, 5, 64, 333])
def test_conv_scan_ragged(ms, dtype, L):
    _check(ms, synth.CONFIGS["m130"].replace(batch=2, dim=40, seqlen=L, dtype=dtype, seed=400 + L), with_prev=True)


@pytest.mark.parametrize("K,silu", [(1, False), (2, True), (3, False), (4, True)])
def test_conv_widths(ms, K, silu):
    _check(ms, synth.CONFIGS["m130"].replace(batch=2, dim=24, seqlen=200, seed=410 + K), K=K, silu=silu)


@pytest.mark.parametrize("N", [8, 32, 64])
def test_conv_state_sizes(ms, N):
    _check(ms, synth.CONFIGS["m130"].replace(batch=2, dim=20, dstate=N, seqlen=150, seed=420 + N))


def test_conv_scan_with_hold(ms):
    _check(ms, synth.CONFIGS["m130"].replace(batch=2, dim=40, seqlen=300, seed=430), disc="zoh")


def test_conv_split_sequence(ms):
    """Few channels, long sequence: the segments of the split time axis read the inputs before
    their first step from the previous segment."""
    _check(ms, synth.CONFIGS["long"].replace(dim=16, seqlen=30000, seed=440), with_prev=True)


def test_conv_pieces_equal_whole(ms):
    """Scanning in two pieces, handing on last_state (as h0) and the last K-1 inputs (as
    conv_prev), gives the one-piece result."""
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=32, seqlen=300, seed=450)
    inp = synth.scan_inputs(cfg)
    cp = synth.conv_params(cfg, 4)
    d = dev_inputs(inp, cfg.dtype)
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    w, cb = f(cp["conv_w"]), f(cp["conv_bias"])
    y_all, st_all = ms.mamba_scan_fwd_conv(d["u"], w, cb, d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                           d["delta_bias"])
    cut = 137
    part = lambda t, a, b: t[..., a:b].contiguous()
    y1, st1 = ms.mamba_scan_fwd_conv(part(d["u"], 0, cut), w, cb, part(d["delta"], 0, cut), d["A"],
                                     part(d["B"], 0, cut), part(d["C"], 0, cut), d["D"], part(d["z"], 0, cut),
                                     d["delta_bias"])
    y2, st2 = ms.mamba_scan_fwd_conv(part(d["u"], cut, None), w, cb, part(d["delta"], cut, None), d["A"],
                                     part(d["B"], cut, None), part(d["C"], cut, None), d["D"],
                                     part(d["z"], cut, None), d["delta_bias"], conv_prev=part(d["u"], cut - 3, cut),
                                     h0=st1)
    torch.cuda.synchronize()
    assert rel_err(from_dev(torch.cat([y1, y2], dim=2)), from_dev(y_all)) <= 1e-5
    assert rel_err(from_dev(st2), from_dev(st_all)) <= 1e-5


def test_conv_full_size_sampled(ms):
    cfg = synth.CONFIGS["m130"]
    inp = synth.scan_inputs(cfg)
    cp = synth.conv_params(cfg, 4)
    y, st = _gpu(ms, inp, cp, cfg.dtype, True)
    rows = sample_rows(cfg.batch * cfg.dim, 24, seed=9)
    y_ref, st_ref = _oracle(inp, cp, cfg.dtype, True, rows=rows)
    assert rel_err(y.reshape(-1, cfg.seqlen)[rows], y_ref) <= TOL[cfg.dtype]
    assert rel_err(st.reshape(-1, cfg.dstate)[rows], st_ref) <= TOL[cfg.dtype]
