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


def test_selective_scan_refuses_wide_state_before_forward(ms):
    x = torch.zeros((1, 4, 16), device="cuda", requires_grad=True)
    A = -torch.ones((4, 32), device="cuda")
    Bm = torch.zeros((1, 32, 16), device="cuda")
    n0 = ms.launch_count()
    with pytest.raises(ValueError, match="d_state <= 16"):
        ms.selective_scan(x, torch.zeros_like(x), A, Bm, Bm.clone())
    assert ms.launch_count() == n0
    with torch.no_grad():  # no gradient wanted: the forward pass runs
        y, _ = ms.selective_scan(x, torch.zeros_like(x), A, Bm, Bm.clone())
    assert y.shape == x.shape
