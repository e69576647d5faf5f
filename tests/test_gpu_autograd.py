"""The autograd operation selective_scan on the GPU: forward through mamba_scan_fwd, backward
through mamba_scan_bwd (states recomputed, visual guide to Mamba and SSMs, section 3.4), with the
gradients autograd delivers compared tensor by tensor with the fp64 gradient oracle.

The loss is sum(dy * y) + sum(dlast * last_state), so the gradients are those the oracle defines
for that loss.  Bounds: max|g_gpu - g_oracle| / max|g_oracle| <= 1e-4 (fp32 storage) and <= 2e-2
(bf16 storage; there the gradients of B and C reach their bf16 inputs rounded to bf16).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, from_dev, rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ms():
    import sequence_scan_selective_b300 as m
    return m


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("with_h0", [False, True])
def test_selective_scan_gradients_match_oracle(ms, dtype, with_h0):
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=40, dstate=16, seqlen=200, dtype=dtype, seed=70)
    inp = synth.scan_inputs(cfg)
    g = synth.grad_inputs(cfg)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    t = {k: to_dev(inp[k], dtype) for k in ("u", "delta", "z", "B", "C")}
    t.update({k: f32(inp[k]) for k in ("A", "D", "delta_bias")})
    t["h0"] = f32(g["h0"]) if with_h0 else None
    for v in t.values():
        if v is not None:
            v.requires_grad_(True)
    y, last = ms.selective_scan(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"],
                                True, h0=t["h0"])
    dy = to_dev(g["dy"], dtype)
    dl = f32(g["dlast"])
    ((y.float() * dy.float()).sum() + (last * dl).sum()).backward()
    torch.cuda.synchronize()
    ms.device_status()
    ref = oracle.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], synth.widen(g["dy"], dtype),
                          inp["D"], inp["z"], inp["delta_bias"], True, dtype,
                          h0=g["h0"] if with_h0 else None, dlast_state=g["dlast"])
    pairs = {"u": "du", "delta": "ddelta", "z": "dz", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "delta_bias": "ddelta_bias", "h0": "dh0"}
    for k, gk in pairs.items():
        if t[k] is None:
            continue
        assert t[k].grad is not None, k
        assert t[k].grad.dtype == t[k].dtype and t[k].grad.shape == t[k].shape, k
        e = rel_err(from_dev(t[k].grad), ref[gk])
        assert e <= TOL[dtype], f"{k}: rel err {e:.3e}"


@pytest.mark.parametrize("N", [32, 64])
def test_selective_scan_wide_state(ms, N):
    """d_state above 16 trains too: the backward pass takes the states in blocks of 16."""
    cfg = synth.CONFIGS["m130"].replace(batch=1, dim=24, dstate=N, seqlen=120, seed=72 + N)
    inp = synth.scan_inputs(cfg)
    g = synth.grad_inputs(cfg)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    t = {k: f32(inp[k]) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias")}
    for v in t.values():
        v.requires_grad_(True)
    y, last = ms.selective_scan(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True)
    ((y * f32(g["dy"])).sum() + (last * f32(g["dlast"])).sum()).backward()
    torch.cuda.synchronize()
    ref = oracle.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], g["dy"].astype(np.float64),
                          inp["D"], inp["z"], inp["delta_bias"], True, "f32", dlast_state=g["dlast"])
    pairs = {"u": "du", "delta": "ddelta", "z": "dz", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "delta_bias": "ddelta_bias"}
    for k, gk in pairs.items():
        e = rel_err(from_dev(t[k].grad), ref[gk])
        assert e <= TOL["f32"], f"{k}: rel err {e:.3e}"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_selective_scan_conv_gradients_match_oracle(ms, dtype):
    """The fused block (causal convolution + scan) as an autograd operation, against the oracle
    chain: oracle convolution (fp64 u), oracle scan gradients on that u, oracle convolution
    gradient."""
    K = 4
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=36, dstate=16, seqlen=300, dtype=dtype, seed=71)
    inp = synth.scan_inputs(cfg)
    g = synth.grad_inputs(cfg)
    cp = synth.conv_params(cfg, K)
    prev = synth.conv_prev(cfg, K)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    t = {k: to_dev(inp[k], dtype) for k in ("u", "delta", "z", "B", "C")}
    t.update({k: f32(inp[k]) for k in ("A", "D", "delta_bias")})
    t.update(conv_w=f32(cp["conv_w"]), conv_bias=f32(cp["conv_bias"]), conv_prev=f32(prev), h0=f32(g["h0"]))
    for v in t.values():
        v.requires_grad_(True)
    y, last = ms.selective_scan_conv(t["u"], t["conv_w"], t["conv_bias"], t["delta"], t["A"], t["B"], t["C"], t["D"],
                                     t["z"], t["delta_bias"], True, conv_prev=t["conv_prev"], h0=t["h0"])
    dy = to_dev(g["dy"], dtype)
    ((y.float() * dy.float()).sum() + (last * f32(g["dlast"])).sum()).backward()
    torch.cuda.synchronize()
    ms.device_status()
    w = lambda a: synth.widen(a, dtype)
    u = oracle.causal_conv(inp["u"], cp["conv_w"], cp["conv_bias"], True, dtype, x_prev=prev)
    ref = oracle.scan_bwd(u, w(inp["delta"]), inp["A"], w(inp["B"]), w(inp["C"]), w(g["dy"]), inp["D"], w(inp["z"]),
                          inp["delta_bias"], True, "f64", h0=g["h0"], dlast_state=g["dlast"])
    cg = oracle.causal_conv_bwd(inp["u"], cp["conv_w"], ref["du"], cp["conv_bias"], True, dtype, x_prev=prev)
    ref.update(dx=cg["dx"], dconv_w=cg["dw"], dconv_bias=cg["dconv_bias"], dconv_prev=cg["dx_prev"])
    pairs = {"u": "dx", "delta": "ddelta", "z": "dz", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "delta_bias": "ddelta_bias", "h0": "dh0", "conv_w": "dconv_w", "conv_bias": "dconv_bias",
             "conv_prev": "dconv_prev"}
    for k, gk in pairs.items():
        assert t[k].grad is not None, k
        assert t[k].grad.dtype == t[k].dtype and t[k].grad.shape == t[k].shape, k
        e = rel_err(from_dev(t[k].grad), ref[gk])
        assert e <= TOL[dtype], f"{k}: rel err {e:.3e}"
