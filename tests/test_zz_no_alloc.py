"""The allocation-free scan entry point (mamba_scan_fwd_noalloc) against the regular one.

Some callers cannot let a library allocate device memory: a process that hands all of it to its own
pool allocator up front, or one that runs under a fixed, audited budget.  For them the library
keeps the carries of a split sequence in a fixed scratch array of its own instead of calling the
CUDA allocator.  These tests call that entry point through the C ABI on shapes that do split the
sequence, and check its results against mamba_scan_fwd's, on two calls in a row (the scratch array
is shared and keeps the previous call's contents).  This file is collected last on purpose.
"""
import ctypes

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


class _DefaultPool:
    """The current device's default memory pool (the one cudaMallocAsync draws from), through the
    driver API: its high-water mark of memory in use, which a test can reset to zero."""

    USED_MEM_HIGH = 8  # CU_MEMPOOL_ATTR_USED_MEM_HIGH

    def __init__(self):
        self.cu = ctypes.CDLL("libcuda.so.1")
        assert self.cu.cuInit(0) == 0
        dev = ctypes.c_int()
        assert self.cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
        self.pool = ctypes.c_void_p()
        assert self.cu.cuDeviceGetDefaultMemPool(ctypes.byref(self.pool), dev) == 0

    def reset_high(self):
        zero = ctypes.c_uint64(0)
        assert self.cu.cuMemPoolSetAttribute(self.pool, self.USED_MEM_HIGH, ctypes.byref(zero)) == 0

    def high(self) -> int:
        v = ctypes.c_uint64(0)
        assert self.cu.cuMemPoolGetAttribute(self.pool, self.USED_MEM_HIGH, ctypes.byref(v)) == 0
        return int(v.value)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_noalloc_matches_regular_entry_point_twice(ms, dtype):
    # 32 channels and 8192 steps: too few channels for the GPU, so the time axis is split into
    # segments and the carries go through the scratch array
    pool = _DefaultPool()
    outs = []
    for call, seed in enumerate((41, 42)):
        cfg = synth.CONFIGS["long"].replace(batch=1, dim=32, seqlen=8192, dtype=dtype, seed=seed)
        d = dev_inputs(synth.scan_inputs(cfg), dtype)
        y_ref = torch.empty_like(d["u"])
        st_ref = torch.empty((cfg.batch, cfg.dim, cfg.dstate), device="cuda")
        y = torch.full_like(y_ref, float("nan"))
        st = torch.full_like(st_ref, float("nan"))
        torch.cuda.synchronize()
        # positive control: the regular entry point takes the carries from the stream-ordered
        # allocator, so the pool's high-water mark rises; two launches show the split ran
        pool.reset_high()
        n0 = ms.launch_count()
        ms.mamba_scan_fwd(*_args(d), y=y_ref, last_state=st_ref)
        torch.cuda.synchronize()
        assert ms.launch_count() - n0 == 2
        assert pool.high() > 0
        pool.reset_high()
        n0 = ms.launch_count()
        ms.mamba_scan_fwd_noalloc(*_args(d), y=y, last_state=st)
        torch.cuda.synchronize()
        assert ms.launch_count() - n0 == 2, "the shape no longer splits the time axis"
        assert pool.high() == 0, "the allocation-free entry point drew memory from the pool"
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


def _header_bound_bytes(batch, dim, N, L, dtype, nsm):
    """The scratch bound include/mamba_scan.h states for a shape: S segments at most, times the
    bytes of one segment's carries (S of them for N <= 16, S - 1 above)."""
    tc = 32 if dtype == "f32" else 64
    smax_len = max(1, L // (8 * tc))
    if N <= 16:
        units = batch * -(-dim // 32)
        S = 1 if units * 2 > 4 * nsm else min(-(-4 * nsm // units) + 1, smax_len)
        nseg_carries = S
    else:
        units = batch * -(-dim // 8)
        S = 1 if units >= 5 * nsm else min(-(-10 * nsm // units), smax_len)
        nseg_carries = S - 1
    return 0 if S <= 1 else nseg_carries * batch * dim * N * 8


@pytest.mark.parametrize("dim,L", [(32, 8192), (64, 65536), (256, 16384), (1536, 32768)])
def test_noalloc_shapes_within_the_stated_bound(ms, dim, L):
    """Shapes whose stated bound fits the fixed scratch are accepted and match the regular entry
    point (the bound is what a caller can compute from the shape and the SM count)."""
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    bound = _header_bound_bytes(1, dim, 16, L, "f32", nsm)
    assert bound <= 4 << 20, bound
    cfg = synth.CONFIGS["long"].replace(batch=1, dim=dim, seqlen=L, seed=50 + dim)
    d = dev_inputs(synth.scan_inputs(cfg), "f32")
    y_ref, st_ref = ms.mamba_scan_fwd(*_args(d))
    y, st = ms.mamba_scan_fwd_noalloc(*_args(d))
    torch.cuda.synchronize()
    assert rel_err(from_dev(y), from_dev(y_ref)) <= TOL["f32"]
    assert rel_err(from_dev(st), from_dev(st_ref)) <= TOL["f32"]
