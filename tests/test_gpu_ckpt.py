"""GPU parity of the forward pass of training (state checkpoints) and of the backward pass that
starts from them.

* mamba_scan_fwd_train gives the same y and last_state as mamba_scan_fwd, bit for bit (the same
  kernels with extra stores), and its checkpoint of slot s is the state after the first 8 s steps:
  the oracle's last state of the sequence cut to 8 s positions.
* mamba_scan_bwd with those checkpoints matches the oracle's gradients with the bounds of the
  backward tests, for both forward kernels, both discretisations and both storage types.
* A sequence the forward planner splits along L gets no checkpoints (None), and a backward pass
  that splits ignores them.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, dev_inputs, from_dev, rel_err, to_dev

pytestmark = pytest.mark.gpu

GRADS = ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0")
STATE_TOL = {"f32": 1e-4, "bf16": 1e-3}  # fp32 states from stored (exactly widened) inputs


@pytest.fixture(scope="module")
def ms():
    import sequence_scan_selective_b300 as m
    return m


class _env:
    def __init__(self, **kv):
        self.kv, self.old = kv, {}

    def __enter__(self):
        for k, v in self.kv.items():
            self.old[k] = os.environ.get(k)
            os.environ[k] = v

    def __exit__(self, *exc):
        for k, v in self.old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _inputs(cfg):
    inp = synth.scan_inputs(cfg)
    g = synth.grad_inputs(cfg)
    inp["dy"], inp["h0"], inp["dlast"] = g["dy"], g["h0"], g["dlast"]
    return inp


def _f32(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def _train(ms, inp, dtype, disc):
    d = dev_inputs(inp, dtype)
    h0 = _f32(inp["h0"])
    y0, st0 = ms.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d.get("D"), d.get("z"),
                                d.get("delta_bias"), True, h0=h0, disc=disc)
    y, st, ck = ms.mamba_scan_fwd_train(d["u"], d["delta"], d["A"], d["B"], d["C"], d.get("D"), d.get("z"),
                                        d.get("delta_bias"), True, h0=h0, disc=disc)
    torch.cuda.synchronize()
    ms.device_status()
    return d, h0, (y0, st0), (y, st, ck)


def _ckpt_states_ok(inp, ck, dtype, disc, slots):
    """Checkpoint s against the oracle's state after the first 8 s steps."""
    N = inp["A"].shape[1]
    got = from_dev(ck)
    for s in slots:
        cut = lambda a: None if a is None else np.ascontiguousarray(a[..., :8 * s])
        _, st = oracle.scan(cut(inp["u"]), cut(inp["delta"]), inp["A"], cut(inp["B"]), cut(inp["C"]), inp["D"],
                            cut(inp["z"]), inp["delta_bias"], True, dtype, h0=inp["h0"], disc=disc)
        err = rel_err(got[:, s, :, :N], st)
        assert err <= STATE_TOL[dtype], (s, err)
    assert not np.any(got[:, 1:, :, N:]), "states past N must be written as zero"


def _bwd_check(ms, inp, d, h0, dtype, disc, ck):
    dy = to_dev(inp["dy"], dtype)
    dl = _f32(inp["dlast"])
    got = ms.mamba_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], dy, d.get("D"), d.get("z"),
                            d.get("delta_bias"), True, h0=h0, dlast_state=dl, disc=disc, ckpt=ck)
    plain = ms.mamba_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], dy, d.get("D"), d.get("z"),
                              d.get("delta_bias"), True, h0=h0, dlast_state=dl, disc=disc)
    torch.cuda.synchronize()
    ms.device_status()
    ref = oracle.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], synth.widen(inp["dy"], dtype),
                          inp["D"], inp["z"], inp["delta_bias"], True, dtype, h0=inp["h0"],
                          dlast_state=inp["dlast"], disc=disc)
    errs = {k: rel_err(from_dev(got[k]), ref[k]) for k in GRADS}
    bad = {k: v for k, v in errs.items() if not v <= TOL[dtype]}
    assert not bad, f"gradients from checkpoints off: {bad} (all: {errs})"
    # and the two backward routes agree more closely than either does with the oracle's rounding
    for k in GRADS:
        assert rel_err(from_dev(got[k]), from_dev(plain[k])) <= TOL[dtype], k


@pytest.mark.parametrize("kernel", ["lane", "warp"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("disc", ["simple", "zoh"])
@pytest.mark.parametrize("L,N", [(77, 16), (200, 5), (512, 13)])
def test_train_checkpoints_and_gradients(ms, kernel, dtype, disc, L, N):
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=40, dstate=N, seqlen=L, dtype=dtype, seed=300 + L + N)
    inp = _inputs(cfg)
    with _env(MAMBA_SCAN_KERNEL=kernel, MAMBA_SCAN_NSEG="1", MAMBA_SCAN_BWD_NSEG="1"):
        d, h0, (y0, st0), (y, st, ck) = _train(ms, inp, dtype, disc)
        assert torch.equal(y, y0) and torch.equal(st, st0), "the training forward pass changed y or the state"
        assert ck is not None and ck.shape == (2, (L + 7) // 8, 40, 16)
        nslot = (L + 7) // 8
        _ckpt_states_ok(inp, ck, dtype, disc, sorted({1, nslot // 2, nslot - 1}))
        _bwd_check(ms, inp, d, h0, dtype, disc, ck)


@pytest.mark.parametrize("kernel", ["lane", "warp"])
def test_train_split_forward_keeps_no_checkpoints(ms, kernel):
    cfg = synth.CONFIGS["m130"].replace(batch=1, dim=32, dstate=16, seqlen=4096, seed=330)
    inp = _inputs(cfg)
    with _env(MAMBA_SCAN_KERNEL=kernel, MAMBA_SCAN_NSEG="3"):
        d, h0, (y0, st0), (y, st, ck) = _train(ms, inp, cfg.dtype, "simple")
        assert ms.train_checkpoint_bytes(d["u"], d["A"]) == 0
        assert ck is None
        assert torch.equal(y, y0) and torch.equal(st, st0)
        # with a buffer given, the library itself reports that it wrote nothing
        buf = torch.full((1, 512, 32, 16), 7.0, device="cuda")
        y2, st2, ck2 = ms.mamba_scan_fwd_train(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                               d["delta_bias"], True, h0=h0, ckpt=buf)
        torch.cuda.synchronize()
        assert ck2 is None and torch.equal(y2, y0) and torch.equal(st2, st0)
        assert bool(torch.all(buf == 7.0)), "a split forward pass wrote checkpoints"


@pytest.mark.parametrize("kernel", ["lane", "warp"])
@pytest.mark.parametrize("nseg", ["1", "2", ""])
def test_train_checkpoint_bytes_matches_what_is_written(ms, kernel, nseg):
    """The size query and the forward pass agree on whether checkpoints are kept, with the
    library's own plan ("") and forced segment counts."""
    cfg = synth.CONFIGS["m130"].replace(batch=1, dim=64, dstate=16, seqlen=4096, seed=360)
    inp = _inputs(cfg)
    d = dev_inputs(inp, cfg.dtype)
    env = {"MAMBA_SCAN_KERNEL": kernel}
    if nseg:
        env["MAMBA_SCAN_NSEG"] = nseg
    with _env(**env):
        nbytes = ms.train_checkpoint_bytes(d["u"], d["A"])
        buf = torch.empty((1, 512, 64, 16), device="cuda")
        _y, _st, ck = ms.mamba_scan_fwd_train(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                              d["delta_bias"], True, ckpt=buf)
        torch.cuda.synchronize()
    assert (ck is not None) == (nbytes > 0)
    assert nbytes in (0, buf.numel() * 4)
    if nseg == "1":
        assert nbytes == buf.numel() * 4


def test_train_checkpoints_ignored_by_a_split_backward(ms):
    cfg = synth.CONFIGS["m130"].replace(batch=1, dim=64, dstate=16, seqlen=2048, seed=340)
    inp = _inputs(cfg)
    with _env(MAMBA_SCAN_NSEG="1", MAMBA_SCAN_BWD_NSEG="3"):
        d, h0, _plain, (_y, _st, ck) = _train(ms, inp, cfg.dtype, "simple")
        assert ck is not None
        _bwd_check(ms, inp, d, h0, cfg.dtype, "simple", ck)


def test_train_wide_state_keeps_no_checkpoints(ms):
    """N > 16: the binding runs the plain forward pass and returns no checkpoints; the library
    itself refuses a checkpoint buffer for that shape."""
    cfg = synth.CONFIGS["m130"].replace(batch=1, dim=8, dstate=17, seqlen=16, seed=350)
    inp = _inputs(cfg)
    d = dev_inputs(inp, cfg.dtype)
    assert ms.train_checkpoint_bytes(d["u"], d["A"]) == 0
    y, st, ck = ms.mamba_scan_fwd_train(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                        d["delta_bias"])
    y0, st0 = ms.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"])
    torch.cuda.synchronize()
    assert ck is None and torch.equal(y, y0) and torch.equal(st, st0)
    with pytest.raises(RuntimeError, match="dstate"):
        ms.mamba_scan_fwd_train(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                                ckpt=torch.empty((1, 2, 8, 16), device="cuda"))


def test_train_full_size_sampled(ms):
    """The 4 x 4096 x 16 x 2048 bf16 layer: checkpoints of sampled channels against the oracle,
    and the backward pass from them against the plain backward pass everywhere."""
    cfg = synth.CONFIGS["b14"]
    inp = _inputs(cfg)
    d, h0, (y0, st0), (y, st, ck) = _train(ms, inp, cfg.dtype, "simple")
    assert torch.equal(y, y0) and torch.equal(st, st0)
    assert ck is not None
    bsz, dim, L, N = cfg.batch, cfg.dim, cfg.seqlen, cfg.dstate
    rows = np.array([0, 1, 777, dim - 1, dim + 5, 3 * dim + 100], dtype=np.int64)
    r = lambda a, w: a.reshape(bsz * dim, w)
    for s in (1, 100, (L + 7) // 8 - 1):
        got = from_dev(ck[:, s])
        cut = lambda a: np.ascontiguousarray(r(a, L)[rows][:, :8 * s])
        bsel = rows // dim
        _, want = oracle.scan_rows(rows, dim, cut(inp["u"]), cut(inp["delta"]), cut(inp["z"]), inp["A"], inp["D"],
                                   inp["delta_bias"], np.ascontiguousarray(inp["B"][..., :8 * s]),
                                   np.ascontiguousarray(inp["C"][..., :8 * s]), True, cfg.dtype,
                                   r(inp["h0"], N)[rows])
        have = got[bsel, rows % dim, :N]
        assert rel_err(have, want) <= STATE_TOL[cfg.dtype], s
    dy = to_dev(inp["dy"], cfg.dtype)
    dl = _f32(inp["dlast"])
    g1 = ms.mamba_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], dy, d["D"], d["z"], d["delta_bias"], True,
                           h0=h0, dlast_state=dl, ckpt=ck)
    g0 = ms.mamba_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], dy, d["D"], d["z"], d["delta_bias"], True,
                           h0=h0, dlast_state=dl)
    torch.cuda.synchronize()
    ms.device_status()
    for k in GRADS:
        assert rel_err(from_dev(g1[k]), from_dev(g0[k])) <= TOL[cfg.dtype], k
