"""The allocation-free scan entry point (mamba_scan_fwd_noalloc) against the regular one.

Some callers cannot let a library allocate device memory: a process that hands all of it to its own
pool allocator up front, or one that runs under a fixed, audited budget.  For them the library
keeps the carries of a split sequence in a fixed scratch array of its own instead of calling the
CUDA allocator.  These tests call that entry point through the C ABI on shapes that do split the
sequence, and check its results against mamba_scan_fwd's, on two calls in a row (the scratch array
is shared and keeps the previous call's contents).  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import TOL, dev_inputs, from_dev, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ms():
    import sequence_scan_selective_b300 as m
    return m


def _args(d):
    return (d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"], True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_noalloc_matches_regular_entry_point_twice(ms, dtype):
    # 32 channels and 8192 steps: too few channels for the GPU, so the time axis is split into
    # segments and the carries go through the scratch array
    outs = []
    for call, seed in enumerate((41, 42)):
        cfg = synth.CONFIGS["long"].replace(batch=1, dim=32, seqlen=8192, dtype=dtype, seed=seed)
        d = dev_inputs(synth.scan_inputs(cfg), dtype)
        y_ref, st_ref = ms.mamba_scan_fwd(*_args(d))
        y = torch.full_like(y_ref, float("nan"))
        st = torch.full_like(st_ref, float("nan"))
        ms.mamba_scan_fwd_noalloc(*_args(d), y=y, last_state=st)
        torch.cuda.synchronize()
        ms.device_status()
        assert rel_err(from_dev(y), from_dev(y_ref)) <= TOL[dtype], f"call {call}"
        assert rel_err(from_dev(st), from_dev(st_ref)) <= TOL[dtype], f"call {call}"
        outs.append(from_dev(y))
    assert not np.array_equal(outs[0], outs[1])  # the second call really computed new inputs


def test_noalloc_unsplit_shape(ms):
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=256, seqlen=512, seed=43)
    d = dev_inputs(synth.scan_inputs(cfg), cfg.dtype)
    y_ref, st_ref = ms.mamba_scan_fwd(*_args(d))
    for _ in range(2):
        y, st = ms.mamba_scan_fwd_noalloc(*_args(d))
        torch.cuda.synchronize()
        assert rel_err(from_dev(y), from_dev(y_ref)) <= TOL["f32"]
        assert rel_err(from_dev(st), from_dev(st_ref)) <= TOL["f32"]


def test_noalloc_rejects_scratch_overflow(ms):
    # a forced split into many segments: the carries of 4096 channels x 64 states then need tens
    # of MB, more than the 4 MB scratch; the size check runs on the host before any launch
    import os
    os.environ["MAMBA_SCAN_NSEG"] = "64"
    try:
        x = torch.zeros((1, 4096, 8192), device="cuda")
        A = -torch.ones((4096, 64), device="cuda")
        Bm = torch.zeros((1, 64, 8192), device="cuda")
        with pytest.raises(ms.MambaScanError, match="scratch"):
            ms.mamba_scan_fwd_noalloc(x, x.clone(), A, Bm, Bm.clone())
    finally:
        os.environ.pop("MAMBA_SCAN_NSEG", None)
