"""GPU parity at the million-token workload: batch 1, d_inner 1536, N 16, L = 2^20, fp32 storage.

The news write-up of the Mamba paper ("architecture" section) and the summary of its claims state
that the selective SSM scales linearly to sequences of a million tokens.  At that length the
channels alone cannot fill the GPU, so the library splits the time axis into segments and
regroups the associative scan operator (visual guide to Mamba and SSMs, section 3.3).  This test
runs the whole workload through mamba_scan_fwd with the launch plan the library chooses by itself
(no test knobs), then compares y over the full length and the final state of sampled channels,
element by element, with the fp64 oracle (fp32 bound: max|y_gpu - y_oracle| / max|y_oracle| <=
1e-4).  The inputs are generated block by block straight into device memory; the oracle's rows
are regenerated on their own (every row has its own random stream, so they are bit-identical).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, from_dev, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ms():
    import sequence_scan_selective_b300 as m
    return m


def _device_inputs(cfg, block=64):
    n, L = cfg.batch * cfg.dim, cfg.seqlen
    d = {k: torch.empty((cfg.batch, cfg.dim, L), device="cuda", dtype=torch.float32) for k in ("u", "delta", "z")}
    for lo in range(0, n, block):
        hi = min(n, lo + block)
        r = synth.scan_rows(cfg, range(lo, hi))
        for k in ("u", "delta", "z"):
            d[k].view(n, L)[lo:hi].copy_(torch.from_numpy(r[k]))
    bc = synth.scan_bc(cfg)
    for k in ("B", "C"):
        d[k] = torch.from_numpy(bc[k]).cuda()
    for k, v in synth.params(cfg).items():
        d[k] = torch.from_numpy(np.ascontiguousarray(v, np.float32)).cuda()
    return d, bc


def test_million_token_workload_full_size(ms):
    cfg = synth.CONFIGS["long"]
    assert (cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen, cfg.dtype) == (1, 1536, 16, 1 << 20, "f32")
    d, bc = _device_inputs(cfg)
    n0 = ms.launch_count()
    y, st = ms.mamba_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"], True)
    launches = ms.launch_count() - n0
    torch.cuda.synchronize()
    ms.device_status()
    # the plan split the time axis (a carry launch before the scan launch)
    assert launches == 2, launches
    for k in ("u", "delta", "z"):
        del d[k]
    # first and last channels, both sides of every multiple of 8 and 32 near the middle and the
    # ends (work-unit and CTA boundaries fall on such multiples), and a few random channels
    rows = sorted({0, 1, 7, 8, 31, 32, 767, 768, 1503, 1504, 1534, 1535}
                  | set(np.random.default_rng(7).choice(cfg.dim, 4, replace=False).tolist()))
    rows = np.array(rows, dtype=np.int64)
    p = synth.params(cfg)
    worst_y = worst_s = 0.0
    for lo in range(0, len(rows), 4):  # 4 channels at a time keeps the fp64 copies small
        rs = rows[lo:lo + 4]
        sub = synth.scan_rows(cfg, rs)
        y_ref, st_ref = oracle.scan_rows(rs, cfg.dim, sub["u"], sub["delta"], sub["z"], p["A"], p["D"],
                                         p["delta_bias"], bc["B"], bc["C"], True, cfg.dtype)
        idx = torch.from_numpy(rs).cuda()
        yg = from_dev(y.view(-1, cfg.seqlen)[idx])
        sg = from_dev(st.view(-1, cfg.dstate)[idx])
        for i, r in enumerate(rs):
            ey, es = rel_err(yg[i], y_ref[i]), rel_err(sg[i], st_ref[i])
            worst_y, worst_s = max(worst_y, ey), max(worst_s, es)
            assert ey <= TOL["f32"], f"channel {r}: y rel err {ey:.3e}"
            assert es <= TOL["f32"], f"channel {r}: state rel err {es:.3e}"
    print(f"million-token workload: worst y rel err {worst_y:.3e}, worst state rel err {worst_s:.3e} "
          f"over {len(rows)} channels")
    del y, st, d
    torch.cuda.empty_cache()
