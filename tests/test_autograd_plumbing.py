"""The autograd wrapper (selective_scan) only routes tensors between the forward and backward entry
points.  Here both entry points are replaced, on the CPU, by stand-ins built from the oracle, and
the gradients autograd hands back are compared with the stand-in's outputs: every gradient must
arrive at its own input, in its input's dtype, with None for absent inputs."""
import numpy as np
import pytest
import torch

import oracle
import synth


@pytest.fixture()
def ms_fake(monkeypatch):
    import sequence_scan_selective_b300 as ms
    calls = {}

    def fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, h0=None, disc="simple", **_):
        n = lambda t: None if t is None else t.detach().numpy()
        y, st = oracle.scan(n(u), n(delta), n(A), n(B), n(C), n(D), n(z), n(delta_bias), softplus, "f32",
                            h0=None if h0 is None else n(h0).astype(np.float64), disc=disc)
        return torch.from_numpy(y.astype(np.float32)), torch.from_numpy(st.astype(np.float32))

    def fwd_train(*args, **kw):  # the training forward pass: also a checkpoint tensor for the backward pass
        y, st = fwd(*args, **kw)
        calls["ckpt"] = torch.zeros(1)
        return y, st, calls["ckpt"]

    def bwd(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, softplus=True, h0=None, dlast_state=None,
            disc="simple", ckpt=None, **_):
        calls["bwd_ckpt"] = ckpt
        n = lambda t: None if t is None else t.detach().numpy()
        g = oracle.scan_bwd(n(u), n(delta), n(A), n(B), n(C), n(dy).astype(np.float64), n(D), n(z), n(delta_bias),
                            softplus, "f32", h0=None if h0 is None else n(h0).astype(np.float64),
                            dlast_state=None if dlast_state is None else n(dlast_state).astype(np.float64),
                            disc=disc, nthreads=1)
        out = {k: (None if v is None else torch.from_numpy(v.astype(np.float32))) for k, v in g.items()}
        if D is None:
            out["dD"] = None
        if delta_bias is None:
            out["ddelta_bias"] = None
        if h0 is None:
            out["dh0"] = None
        calls["bwd"] = out
        return out

    monkeypatch.setattr(ms, "mamba_scan_fwd", fwd)
    monkeypatch.setattr(ms, "mamba_scan_fwd_train", fwd_train)
    monkeypatch.setattr(ms, "mamba_scan_bwd", bwd)
    return ms, calls


@pytest.mark.parametrize("drop", [(), ("z", "D"), ("delta_bias", "h0")])
def test_gradients_reach_their_inputs(ms_fake, drop):
    ms, calls = ms_fake
    cfg = synth.CONFIGS["tiny"].replace(batch=2, dim=3, dstate=4, seqlen=9, seed=60)
    inp = synth.scan_inputs(cfg)
    inp["h0"] = np.random.default_rng(61).standard_normal((2, 3, 4)).astype(np.float32)
    names = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias", "h0")
    t = {k: (None if k in drop else torch.from_numpy(np.ascontiguousarray(inp[k])).requires_grad_(True))
         for k in names}
    y, last = ms.selective_scan(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"],
                                True, h0=t["h0"])
    rng = np.random.default_rng(62)
    dy = torch.from_numpy(rng.standard_normal(y.shape).astype(np.float32))
    dl = torch.from_numpy(rng.standard_normal(last.shape).astype(np.float32))
    ((y * dy).sum() + (last * dl).sum()).backward()
    g = calls["bwd"]
    pairs = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "z": "dz",
             "delta_bias": "ddelta_bias", "h0": "dh0"}
    for k, gk in pairs.items():
        if t[k] is None:
            continue
        assert t[k].grad is not None, k
        assert t[k].grad.dtype == t[k].dtype and t[k].grad.shape == t[k].shape, k
        assert torch.equal(t[k].grad, g[gk]), k
    # d_state <= 16: the training forward pass's checkpoints reach the backward pass
    assert calls["bwd_ckpt"] is calls["ckpt"]
