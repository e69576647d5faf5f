"""GPU parity of the fused forward scan against the fp64 oracle, through the C ABI.

Tolerance (fixed for this method): max|y_gpu - y_oracle| / max|y_oracle| <= 1e-4 with fp32 storage
and <= 2e-2 with bf16 storage (fp32 state either way); final states under the same bounds.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, dev_inputs, from_dev, oracle_scan_full, rel_err, sample_rows

pytestmark = pytest.mark.gpu


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


def _run_gpu(ms, d, softplus=True, with_state=True):
    y, st = ms.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d.get("D"), d.get("z"),
                              d.get("delta_bias"), softplus, want_state=with_state)
    torch.cuda.synchronize()
    ms.device_status()
    return y, st


def _check_full(ms, cfg, softplus=True, drop=(), env=None):
    inp = synth.scan_inputs(cfg)
    for k in drop:
        inp[k] = None
    with _env(**(env or {})):
        y, st = _run_gpu(ms, dev_inputs(inp, cfg.dtype), softplus)
    y_ref, st_ref = oracle_scan_full(inp, cfg.dtype, softplus)
    ey, es = rel_err(from_dev(y), y_ref), rel_err(from_dev(st), st_ref)
    assert ey <= TOL[cfg.dtype], f"y rel err {ey:.3e}"
    assert es <= TOL[cfg.dtype], f"state rel err {es:.3e}"
    return ey, es


# The two forward kernels: "lane" (one channel per lane, N <= 16, the default where it applies)
# and "warp" (four lanes per channel, any N; also the exact hold and the fused convolution).
KERNELS = ["lane", "warp"]


def _kenv(kernel, **kv):
    return dict(MAMBA_SCAN_KERNEL=kernel, **kv)


@pytest.mark.parametrize("kernel", KERNELS)
def test_tiny_workload(ms, kernel):
    _check_full(ms, synth.CONFIGS["tiny"], env=_kenv(kernel))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("L", [1, 7, 32, 77, 200, 1000])
def test_ragged_lengths(ms, kernel, dtype, L):
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=40, seqlen=L, dtype=dtype, seed=10 + L)
    _check_full(ms, cfg, env=_kenv(kernel))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("N", [1, 3, 4, 8, 9, 15, 16, 17, 32, 33, 64])
def test_state_sizes(ms, kernel, N):
    if kernel == "lane" and N > 16:
        pytest.skip("the channel-per-lane kernel holds at most 16 states per lane")
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=35, dstate=N, seqlen=160, seed=20 + N)
    _check_full(ms, cfg, env=_kenv(kernel))


def test_default_kernel_for_wide_state(ms):
    """Without a forced kernel, N > 16 takes the four-lanes-per-channel kernel."""
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=35, dstate=24, seqlen=160, seed=19)
    _check_full(ms, cfg)


def test_lane_kernel_refuses_what_it_cannot_do(ms):
    x = torch.zeros((1, 4, 32), device="cuda")
    with _env(MAMBA_SCAN_KERNEL="lane"), pytest.raises(ms.MambaScanError, match="N <= 16"):
        ms.mamba_scan_fwd(x, x.clone(), -torch.ones((4, 32), device="cuda"), torch.zeros((1, 32, 32), device="cuda"),
                          torch.zeros((1, 32, 32), device="cuda"))


@pytest.mark.parametrize("kernel,wmax,stages", [("warp", "1", "2"), ("warp", "3", "3"), ("warp", "15", "4"),
                                                ("warp", "0", "2"), ("lane", "1", "2"), ("lane", "2", "3"),
                                                ("lane", "4", "2"), ("lane", "0", "4")])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tiling_variants(ms, kernel, wmax, stages, dtype):
    """Consumer warps per CTA (work units per CTA) and ring depth change only the schedule."""
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=130, seqlen=333, dtype=dtype, seed=21)
    _check_full(ms, cfg, env=_kenv(kernel, MAMBA_SCAN_WMAX=wmax, MAMBA_SCAN_STAGES=stages))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("drop", [("z",), ("D",), ("delta_bias",), ("z", "D", "delta_bias")])
def test_optional_inputs(ms, kernel, drop):
    cfg = synth.CONFIGS["m130"].replace(batch=3, dim=33, seqlen=96, seed=5)
    _check_full(ms, cfg, drop=drop, env=_kenv(kernel))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_softplus_off(ms, kernel, dtype):
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=32, seqlen=128, dtype=dtype, seed=6)
    inp = synth.scan_inputs(cfg)
    # without softplus the raw delta must itself be a valid step size: |delta| scaled down
    dl = (np.abs(synth.widen(inp["delta"], dtype)) * 0.01).astype(np.float32)
    inp["delta"] = synth.f32_to_bf16_bits(dl) if dtype == "bf16" else dl
    inp["delta_bias"] = np.zeros_like(inp["delta_bias"])
    with _env(**_kenv(kernel)):
        y, st = _run_gpu(ms, dev_inputs(inp, dtype), softplus=False)
    y_ref, st_ref = oracle_scan_full(inp, dtype, softplus=False)
    assert rel_err(from_dev(y), y_ref) <= TOL[dtype]
    assert rel_err(from_dev(st), st_ref) <= TOL[dtype]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_unaligned_rows_take_plain_load_path(ms, kernel, dtype):
    # L * element size not a multiple of 16 bytes: no TMA descriptor is possible for these rows
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=36, seqlen=301, dtype=dtype, seed=7)
    _check_full(ms, cfg, env=_kenv(kernel))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_forced_plain_loads_match(ms, kernel, dtype):
    cfg = synth.CONFIGS["b14"].replace(batch=2, dim=64, seqlen=256, dtype=dtype, seed=8)
    _check_full(ms, cfg, env=_kenv(kernel, MAMBA_SCAN_NO_TMA="1"))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("nseg", [2, 3, 7])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_split_time_axis(ms, kernel, nseg, dtype):
    """Splitting L into segments (carry pass + per-segment scan) regroups the associative scan
    operator (guide section 3.3); results must stay within tolerance of the oracle."""
    cfg = synth.CONFIGS["long"].replace(batch=2, dim=24, seqlen=4000, dtype=dtype, seed=9)
    _check_full(ms, cfg, env=_kenv(kernel, MAMBA_SCAN_NSEG=str(nseg)))


@pytest.mark.parametrize("kernel", KERNELS)
def test_split_with_plain_loads(ms, kernel):
    cfg = synth.CONFIGS["long"].replace(batch=1, dim=40, seqlen=3001, seed=11)
    _check_full(ms, cfg, env=_kenv(kernel, MAMBA_SCAN_NSEG="3"))


@pytest.mark.parametrize("kernel", KERNELS)
def test_segment_count_invariance(ms, kernel):
    cfg = synth.CONFIGS["long"].replace(batch=1, dim=32, seqlen=8192, seed=12)
    d = dev_inputs(synth.scan_inputs(cfg), cfg.dtype)
    outs = []
    for nseg in ("1", "4", "16"):
        with _env(**_kenv(kernel, MAMBA_SCAN_NSEG=nseg)):
            y, st = _run_gpu(ms, d)
        outs.append((from_dev(y), from_dev(st)))
    for y, st in outs[1:]:
        assert rel_err(y, outs[0][0]) <= 1e-5
        assert rel_err(st, outs[0][1]) <= 1e-5


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_split_without_decay(ms, kernel, dtype):
    """States with A = 0 never forget: the state carried into a later segment reaches every one
    of its outputs, so the channel-per-lane split must carry it through the whole segment (no
    early stop), alongside decaying states in the same lanes."""
    cfg = synth.CONFIGS["long"].replace(batch=1, dim=40, seqlen=6000, dtype=dtype, seed=26)
    inp = synth.scan_inputs(cfg)
    inp["A"] = inp["A"].copy()
    inp["A"][:, :3] = 0.0
    inp["A"][5, :] = 0.0  # one channel with no decay at all
    y_ref, st_ref = oracle_scan_full(inp, dtype, True)
    with _env(**_kenv(kernel, MAMBA_SCAN_NSEG="4")):
        y, st = _run_gpu(ms, dev_inputs(inp, dtype))
    assert rel_err(from_dev(y), y_ref) <= TOL[dtype]
    assert rel_err(from_dev(st), st_ref) <= TOL[dtype]


@pytest.mark.parametrize("kernel", KERNELS)
def test_split_large_initial_state(ms, kernel):
    """A large initial state dominates the early outputs of every segment it reaches; the split
    must match the oracle there too (the carried-in part is dropped only once it has decayed far
    below the outputs' resolution)."""
    cfg = synth.CONFIGS["long"].replace(batch=2, dim=36, seqlen=5000, seed=27)
    inp = synth.scan_inputs(cfg)
    inp["A"] = inp["A"].copy()
    inp["A"][:, ::2] *= 0.02  # slow decay: the carry reaches far into the following segments
    h0 = (np.random.default_rng(27).standard_normal((cfg.batch, cfg.dim, cfg.dstate)) * 1e3).astype(np.float32)
    y_ref, st_ref = oracle.scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                inp["delta_bias"], True, cfg.dtype, h0=h0.astype(np.float64))
    d = dev_inputs(inp, cfg.dtype)
    with _env(**_kenv(kernel, MAMBA_SCAN_NSEG="5")):
        y, st = ms.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"], True,
                                  h0=torch.from_numpy(h0).cuda())
        torch.cuda.synchronize()
        ms.device_status()
    assert rel_err(from_dev(y), y_ref) <= TOL["f32"]
    assert rel_err(from_dev(st), st_ref) <= TOL["f32"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_kernels_agree(ms, dtype):
    """Both forward kernels compute the same scan (to rounding) on a shape several CTAs wide."""
    cfg = synth.CONFIGS["b14"].replace(batch=3, dim=300, seqlen=700, dtype=dtype, seed=25)
    d = dev_inputs(synth.scan_inputs(cfg), dtype)
    outs = {}
    for k in KERNELS:
        with _env(MAMBA_SCAN_KERNEL=k):
            outs[k] = [from_dev(t) for t in _run_gpu(ms, d)]
    for k in KERNELS[1:]:
        assert rel_err(outs[k][0], outs["lane"][0]) <= TOL[dtype]
        assert rel_err(outs[k][1], outs["lane"][1]) <= 1e-5


def test_bounded_wait_runs_out(ms):
    """Failure detection on the device: with the test knob the consumer warps of the forward
    kernel wait on a barrier that nothing arrives on, and every wait on another warp is limited to
    1 ms.  The waits run out, the kernel returns (after its copies in flight have landed), the
    status word reports a timeout, and the next call on the same context is correct again."""
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=70, seqlen=512, seed=26)
    inp = synth.scan_inputs(cfg)
    d = dev_inputs(inp, cfg.dtype)
    ms.device_status()  # clear
    with _env(MAMBA_SCAN_KERNEL="lane", MAMBA_SCAN_TEST_STALL="1"):
        ms.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"], True)
        with pytest.raises(ms.MambaScanError) as ei:
            ms.device_status()
    assert ei.value.code == ms.MAMBA_ERR_TIMEOUT
    ms.device_status()  # the word was cleared by the read
    y, st = _run_gpu(ms, d)
    y_ref, st_ref = oracle_scan_full(inp, cfg.dtype)
    assert rel_err(from_dev(y), y_ref) <= TOL["f32"]
    assert rel_err(from_dev(st), st_ref) <= TOL["f32"]


def test_zero_length(ms):
    d = {k: torch.zeros((2, 8, 0), device="cuda") for k in ("u", "delta", "z")}
    st = torch.full((2, 8, 4), 7.0, device="cuda")
    ms.mamba_scan_fwd(d["u"], d["delta"], -torch.ones((8, 4), device="cuda"), torch.zeros((2, 4, 0), device="cuda"),
                      torch.zeros((2, 4, 0), device="cuda"), last_state=st)
    torch.cuda.synchronize()
    assert torch.all(st == 0)


def test_delta_zero_gives_skip_only(ms):
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=20, seqlen=64, seed=13)
    inp = synth.scan_inputs(cfg)
    inp["delta"][:] = 0.0
    inp["delta_bias"][:] = 0.0
    y, st = _run_gpu(ms, dev_inputs(inp, cfg.dtype), softplus=False)
    assert torch.all(st == 0)
    y_ref, _ = oracle_scan_full(inp, cfg.dtype, softplus=False)
    assert rel_err(from_dev(y), y_ref) <= 1e-6


def test_linearity_in_u(ms):
    """Doubling u doubles y exactly (every product scales by a power of two)."""
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=32, seqlen=256, seed=14)
    d = dev_inputs(synth.scan_inputs(cfg), cfg.dtype)
    y1, _ = _run_gpu(ms, d)
    y2, _ = _run_gpu(ms, dict(d, u=d["u"] * 2.0))
    assert rel_err(from_dev(y2), 2.0 * from_dev(y1)) <= 1e-6


def test_bad_arguments_raise(ms):
    x = torch.zeros((1, 4, 16), device="cuda")
    A = -torch.ones((4, 4), device="cuda")
    Bm = torch.zeros((1, 4, 16), device="cuda")
    with pytest.raises(ms.MambaScanError):   # y aliases u
        ms.mamba_scan_fwd(x, x.clone(), A, Bm, Bm.clone(), y=x)
    with pytest.raises(ms.MambaScanError):   # too many states
        ms.mamba_scan_fwd(torch.zeros((1, 4, 16), device="cuda"), torch.zeros((1, 4, 16), device="cuda"),
                          -torch.ones((4, 65), device="cuda"), torch.zeros((1, 65, 16), device="cuda"),
                          torch.zeros((1, 65, 16), device="cuda"))


# ------------------------------------------------------------------------------ full-size workloads
def _check_sampled(ms, cfg, nsample, seed=0, env=None):
    inp = synth.scan_inputs(cfg)
    with _env(**(env or {})):
        y, st = _run_gpu(ms, dev_inputs(inp, cfg.dtype))
    rows = sample_rows(cfg.batch * cfg.dim, nsample, seed)
    sub = {k: inp[k].reshape(cfg.batch * cfg.dim, cfg.seqlen)[rows] for k in ("u", "delta", "z")}
    y_ref, st_ref = oracle.scan_rows(rows, cfg.dim, sub["u"], sub["delta"], sub["z"], inp["A"], inp["D"],
                                     inp["delta_bias"], inp["B"], inp["C"], True, cfg.dtype)
    idx = torch.from_numpy(rows).cuda()
    yg = from_dev(y.reshape(cfg.batch * cfg.dim, cfg.seqlen)[idx])
    sg = from_dev(st.reshape(cfg.batch * cfg.dim, cfg.dstate)[idx])
    ey, es = rel_err(yg, y_ref), rel_err(sg, st_ref)
    assert ey <= TOL[cfg.dtype], f"y rel err {ey:.3e}"
    assert es <= TOL[cfg.dtype], f"state rel err {es:.3e}"


@pytest.mark.parametrize("kernel", KERNELS)
def test_mamba130m_layer_full_size(ms, kernel):
    _check_sampled(ms, synth.CONFIGS["m130"], 192, env=_kenv(kernel))


@pytest.mark.parametrize("kernel", KERNELS)
def test_mamba14b_layer_full_size(ms, kernel):
    _check_sampled(ms, synth.CONFIGS["b14"], 192, env=_kenv(kernel))


def test_wide_state_many_channels(ms):
    """N = 64 with many channels: the plan caps warps per CTA so the tiles fit in shared memory."""
    cfg = synth.CONFIGS["m130"].replace(batch=1, dim=2048, dstate=64, seqlen=256, seed=15)
    _check_full(ms, cfg)


# ------------------------------------------------------------------------------ initial state
@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_initial_state_matches_oracle(ms, kernel, dtype):
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=70, seqlen=300, dtype=dtype, seed=40)
    inp = synth.scan_inputs(cfg)
    h0 = np.random.default_rng(40).standard_normal((cfg.batch, cfg.dim, cfg.dstate)).astype(np.float32)
    d = dev_inputs(inp, dtype)
    with _env(MAMBA_SCAN_KERNEL=kernel):
        y, st = ms.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"], True,
                                  h0=torch.from_numpy(h0).cuda())
    torch.cuda.synchronize()
    y_ref, st_ref = oracle.scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                inp["delta_bias"], True, dtype, h0=h0.astype(np.float64))
    assert rel_err(from_dev(y), y_ref) <= TOL[dtype]
    assert rel_err(from_dev(st), st_ref) <= TOL[dtype]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", ["wide", "split"])
def test_chunked_prefill_in_place(ms, kernel, dtype, shape):
    """A sequence scanned in pieces, each piece continuing from the state the previous one left in
    the same buffer (h0 is last_state), gives the scan of the whole sequence (the recurrence only
    carries h across positions, visual guide section 2.4)."""
    if shape == "wide":
        cfg = synth.CONFIGS["m130"].replace(batch=2, dim=64, seqlen=960, dtype=dtype, seed=41)
        cuts = [0, 320, 653, 960]          # the middle piece has a ragged length
    else:                                   # few channels: every piece is split along L internally
        cfg = synth.CONFIGS["long"].replace(batch=1, dim=32, seqlen=12000, dtype=dtype, seed=42)
        cuts = [0, 4000, 8001, 12000]
    inp = synth.scan_inputs(cfg)
    d = dev_inputs(inp, dtype)
    state = torch.zeros((cfg.batch, cfg.dim, cfg.dstate), device="cuda")
    ys = []
    with _env(MAMBA_SCAN_KERNEL=kernel):
        for a_, b_ in zip(cuts[:-1], cuts[1:]):
            piece = lambda k: d[k][:, :, a_:b_].contiguous()
            y, _ = ms.mamba_scan_fwd(piece("u"), piece("delta"), d["A"], piece("B"), piece("C"), d["D"], piece("z"),
                                     d["delta_bias"], True, h0=state, last_state=state)
            ys.append(y)
    torch.cuda.synchronize()
    ms.device_status()
    y_ref, st_ref = oracle_scan_full(inp, dtype)
    assert rel_err(from_dev(torch.cat(ys, dim=2)), y_ref) <= TOL[dtype]
    assert rel_err(from_dev(state), st_ref) <= TOL[dtype]


def test_initial_state_empty_sequence(ms):
    h0 = torch.randn((2, 8, 4), device="cuda")
    st = torch.full((2, 8, 4), 7.0, device="cuda")
    z = torch.zeros((2, 8, 0), device="cuda")
    ms.mamba_scan_fwd(z, z.clone(), -torch.ones((8, 4), device="cuda"), torch.zeros((2, 4, 0), device="cuda"),
                      torch.zeros((2, 4, 0), device="cuda"), h0=h0, last_state=st)
    torch.cuda.synchronize()
    assert torch.equal(st, h0)


def test_initial_state_partial_overlap_rejected(ms):
    buf = torch.zeros((2 * 8 * 4 + 4,), device="cuda")
    h0, st = buf[:64].view(2, 8, 4), buf[4:68].view(2, 8, 4)
    x = torch.zeros((2, 8, 16), device="cuda")
    with pytest.raises(ms.MambaScanError, match="same buffer"):
        ms.mamba_scan_fwd(x, x.clone(), -torch.ones((8, 4), device="cuda"), torch.zeros((2, 4, 16), device="cuda"),
                          torch.zeros((2, 4, 16), device="cuda"), h0=h0, last_state=st)
