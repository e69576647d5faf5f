"""GPU parity of the backward pass of the scan with the block's causal convolution in front of it
(mamba_scan_bwd_conv) against the fp64 oracle chain: the oracle's convolution gives u in fp64, the
oracle's scan gradients run on that u, and the oracle's convolution gradient takes du back to x.

Every gradient is compared as max|g_gpu - g_oracle| / max|g_oracle| per tensor with the backward
pass's bounds: 1e-4 with fp32 storage, 2e-2 with bf16 storage (the library keeps u and du in the
storage type between its kernels; the oracle keeps them in fp64).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, dev_inputs, from_dev, rel_err, to_dev

pytestmark = pytest.mark.gpu

GRADS = ("dx", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0", "dconv_w", "dconv_bias", "dconv_prev")


@pytest.fixture(scope="module")
def ms():
    import sequence_scan_selective_b300 as m
    return m


def _f32(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def _run(ms, cfg, K, silu, with_prev, disc="simple"):
    dt = cfg.dtype
    inp = synth.scan_inputs(cfg)
    g = synth.grad_inputs(cfg)
    cp = synth.conv_params(cfg, K)
    prev = synth.conv_prev(cfg, K) if with_prev and K > 1 else None
    d = dev_inputs(inp, dt)
    got = ms.mamba_scan_bwd_conv(d["u"], _f32(cp["conv_w"]), _f32(cp["conv_bias"]), d["delta"], d["A"], d["B"],
                                 d["C"], to_dev(g["dy"], dt), d["D"], d["z"], d["delta_bias"], True, conv_silu=silu,
                                 conv_prev=_f32(prev), h0=_f32(g["h0"]), dlast_state=_f32(g["dlast"]), disc=disc)
    torch.cuda.synchronize()
    ms.device_status()
    got = {k: (None if v is None else from_dev(v)) for k, v in got.items()}

    w = lambda a: None if a is None else synth.widen(a, dt)
    u = oracle.causal_conv(inp["u"], cp["conv_w"], cp["conv_bias"], silu, dt, x_prev=prev)
    sg = oracle.scan_bwd(u, w(inp["delta"]), inp["A"], w(inp["B"]), w(inp["C"]), w(g["dy"]), inp["D"], w(inp["z"]),
                         inp["delta_bias"], True, "f64", h0=g["h0"], dlast_state=g["dlast"], disc=disc)
    cg = oracle.causal_conv_bwd(inp["u"], cp["conv_w"], sg["du"], cp["conv_bias"], silu, dt, x_prev=prev)
    ref = dict(sg)
    ref.update(dx=cg["dx"], dconv_w=cg["dw"], dconv_bias=cg["dconv_bias"], dconv_prev=cg["dx_prev"] if K > 1 else None)
    errs = {k: rel_err(got[k], ref[k]) for k in GRADS if got.get(k) is not None and ref.get(k) is not None}
    bad = {k: v for k, v in errs.items() if not v <= TOL[dt]}
    assert not bad, f"gradients off: {bad} (all: {errs})"
    return errs


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("L", [1, 77, 1000, 2500])
def test_conv_bwd_ragged(ms, dtype, L):
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=40, seqlen=L, dtype=dtype, seed=300 + L)
    _run(ms, cfg, 4, True, True)


@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("silu", [True, False])
def test_conv_bwd_widths(ms, K, silu):
    cfg = synth.CONFIGS["m130"].replace(batch=1, dim=24, seqlen=300, seed=310 + K)
    _run(ms, cfg, K, silu, True)


def test_conv_bwd_without_previous_inputs(ms):
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=33, seqlen=500, seed=320)
    _run(ms, cfg, 4, True, False)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv_bwd_with_hold(ms, dtype):
    cfg = synth.CONFIGS["m130"].replace(batch=1, dim=32, seqlen=640, dtype=dtype, seed=330)
    _run(ms, cfg, 4, True, True, disc="zoh")


def test_conv_bwd_empty_sequence(ms):
    """L = 0: the convolution gradients are zeros and the state gradient passes through."""
    dim, N, K = 8, 16, 4
    A = -torch.ones((dim, N), device="cuda")
    w = torch.ones((dim, K), device="cuda")
    e = torch.zeros((1, dim, 0), device="cuda")
    bc = torch.zeros((1, N, 0), device="cuda")
    dl = torch.randn((1, dim, N), device="cuda")
    out = ms.mamba_scan_bwd_conv(e, w, torch.zeros(dim, device="cuda"), e.clone(), A, bc, bc.clone(), e.clone(),
                                 h0=torch.zeros((1, dim, N), device="cuda"), dlast_state=dl)
    torch.cuda.synchronize()
    assert float(out["dconv_w"].abs().max()) == 0.0
    assert float(out["dconv_bias"].abs().max()) == 0.0
    assert float(out["dconv_prev"].abs().max()) == 0.0
    assert torch.equal(out["dh0"], dl)
