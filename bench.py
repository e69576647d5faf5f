#!/usr/bin/env python
"""Throughput of the selective-scan hot path on B300.

One step = one pass of the whole path over one batch of the workload: the fused forward scan over
the sequence (Delta map, discretisation, recurrence, readout, skip, gate, final state) followed by
one recurrent decode step that continues from the scan's final state.  Default workload: the
Mamba-1.4B layer shape (batch 4, d_inner 4096, N 16, L 2048, bf16 inputs, fp32 state); `--workload
m130` selects the Mamba-130M layer shape (batch 8, d_inner 1536, fp32).  The default line also
times the million-token scan (batch 1, d_inner 1536, N 16, L 2^20, fp32) and reports its
per-element rate next to the main workload's scan rate (`long_sequence`).

Prints one JSON line (rank 0).  `value` = elements (batch * d_inner * (L + 1)) per second over all
ranks, device-timed with CUDA events, inputs resident in HBM; the timed steps follow the warm-up
steps and an untimed settle phase (`--settle-ms`, reported as `clock_settle`).  `--pass bwd` times
the backward pass instead and, for N <= 16, the training step both ways (`train_step`: forward +
backward recomputing the checkpoints, or the training forward pass keeping them).  `e2e` = the same metric through the
public API with the inputs copied from pinned host memory and the outputs read back inside the
timed region.  `--impl reference` times the fp64 CPU oracle on the host cores instead.

Multi-GPU (torchrun): every rank runs an independent replica of the workload on its own GPU (the
channels of a scan are independent, so the work shards with no collective); `scaling` is "weak".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

FALLBACK_HBM_GBS = 6400.0
METRIC = "selective-scan elements (batch*d_inner*L)/s"
WORKLOADS = {
    "m130": "Mamba-130M layer scan+decode: batch 8, d_inner 1536, N 16, L 2048, fp32",
    "b14": "Mamba-1.4B layer scan+decode: batch 4, d_inner 4096, N 16, L 2048, bf16 in, fp32 state",
    "long": "million-token scan+decode: batch 1, d_inner 1536, N 16, L 1048576, fp32",
    "decode": "decode steps: batch 128, d_inner 5120, N 16, bf16 in, fp32 state (consecutive tokens)",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--settle-ms", type=float, default=300.0,
                    help="after the warm-up steps, further untimed steps until this much device time has "
                         "passed, so that the timed region does not measure the clocks' ramp from idle")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="b14")
    ap.add_argument("--no-long", action="store_true",
                    help="skip the million-token scan that the b14 and m130 lines report beside their own rate")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pass", dest="which", choices=["fwd", "bwd"], default="fwd",
                    help="fwd: forward scan + decode step (default); bwd: the backward pass alone")
    ap.add_argument("--conv", type=int, default=0,
                    help="fwd pass: fuse a causal depthwise convolution of this width (1-4) in front of the scan")
    ap.add_argument("--disc", choices=["simple", "zoh"], default="simple",
                    help="discretisation of B in the forward scan and decode step")
    ap.add_argument("--seqlen", type=int, default=0,
                    help="override the workload's sequence length (smaller cases of the same shape, e.g. for "
                         "profiling under a size limit)")
    ap.add_argument("--kernel", choices=["auto", "lane", "warp"], default="auto",
                    help="forward scan kernel: the library's choice, one channel per lane, or four lanes per channel")
    ap.add_argument("--decode-inputs", type=int, default=200,
                    help="decode workload: distinct pre-generated steps of inputs, cycled")
    ap.add_argument("--decode-states", type=int, default=6,
                    help="decode workload: state buffers cycled in the second timing (their total is "
                         "kept above twice the L2 size, so the state streams from HBM)")
    return ap.parse_args()


def esize(dtype: str) -> int:
    return 2 if dtype == "bf16" else 4


def scan_bytes(cfg) -> int:
    """Algorithmic bytes of one forward scan: u, delta, z read, y written, B and C read once per
    batch row, A/D/bias read, final state written (Abar, Bbar and h are never stored)."""
    s = esize(cfg.dtype)
    b, d, n, L = cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen
    return b * d * L * 4 * s + 2 * b * n * L * s + d * (n + 2) * 4 + b * d * n * 4


def step_bytes(cfg) -> int:
    """Algorithmic bytes of one decode step: state read + written, x/delta/z read, y written,
    B and C read, A/D/bias read."""
    s = esize(cfg.dtype)
    b, d, n = cfg.batch, cfg.dim, cfg.dstate
    return 2 * b * d * n * 4 + b * d * 4 * s + 2 * b * n * s + d * (n + 2) * 4


def bwd_bytes(cfg) -> int:
    """Algorithmic bytes of one backward pass: u, delta, z, dy read and du, ddelta, dz written per
    element; B, C read and dB, dC (fp32) written per batch row; A, D, bias read and their
    gradients written; h0 and the last-state gradient read, dh0 written.  The state checkpoints of
    the recomputation are not counted."""
    s = esize(cfg.dtype)
    b, d, n, L = cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen
    return b * d * L * 7 * s + b * n * L * (2 * s + 2 * 4) + 2 * d * (n + 2) * 4 + 3 * b * d * n * 4


# FP32 arithmetic floor of the scan: per state-update the recurrence needs 4 FP32 lane operations
# (Delta A, (Delta u) B, Abar h + ..., C.h accumulation; an FMA counts once) and one exp2.  The
# FP32 pipe does 128 lane operations per clock per SM (32 exp2 per clock per SM on the MUFU pipe,
# measured, so both pipes give the same floor); B300: 148 SMs at 2032 MHz at most.
ALU_OPS_PER_STATE_UPDATE = 4
ALU_PEAK_TOPS = 128 * 148 * 2.032e9 / 1e12


def alu_context(cfg, kernel_ms):
    """The forward scan's FP32 arithmetic against the FP32 pipe's peak (context beside the HBM
    roofline: for these shapes the arithmetic floor lies above the HBM floor)."""
    ops = ALU_OPS_PER_STATE_UPDATE * cfg.batch * cfg.dim * cfg.seqlen * cfg.dstate
    achieved = ops / (kernel_ms * 1e-3) / 1e12
    return {"achieved": round(achieved, 2), "peak": round(ALU_PEAK_TOPS, 2), "unit": "Top/s",
            "frac": round(achieved / ALU_PEAK_TOPS, 4), "ops_per_launch": ops,
            "peak_source": "derived: 128 FP32 lanes/clk/SM x 148 SMs x 2032 MHz",
            "floor_us": round(ops / (ALU_PEAK_TOPS * 1e12) * 1e6, 1)}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


# the sources each profiled kernel and the host code that plans its launches are built from
KERNEL_SOURCES = {
    "scan_fwd": ("ptx.cuh", "common.cuh", "scan_fwd.cuh", "fwd_common.cuh", "fwd_warp.cuh", "fwd_warp_f32.cu",
                 "fwd_warp_bf16.cu"),
    "scan_fwd_cl": ("ptx.cuh", "common.cuh", "scan_fwd.cuh", "scan_fwd_cl.cuh", "scan_fix.cuh", "fwd_common.cuh",
                    "fwd_lane.cuh", "fwd_lane_f32.cu", "fwd_lane_bf16.cu"),
    "state_step": ("ptx.cuh", "common.cuh", "state_step.cuh", "step.cu"),
    "scan_bwd": ("ptx.cuh", "common.cuh", "scan_bwd.cuh", "bwd.cu"),
}
KERNEL_SOURCES["scan_fix"] = KERNEL_SOURCES["scan_fwd_cl"]


def source_hash(kernel: str = "scan_fwd") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sequence_scan_selective_b300", "csrc")
    for name in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, kernel: str = "scan_fwd"):
    """DRAM bytes per launch of the kernel from the committed ncu record, if it was taken on the
    current kernel sources; otherwise None."""
    try:
        with open(os.path.join(ROOT, "profiles", f"{kernel}_{workload}.json")) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("source_hash") != source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------------------------------ clocks
class _Nvml:
    """The few NVML calls the sampler needs, through ctypes on the driver's libnvidia-ml."""

    def __init__(self, bus_id: str):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus_id.encode(), ctypes.byref(self.h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByPciBusId_v2 failed")
        self.reason_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sm_clock(self, maximum=False) -> int:
        v = self.ct.c_uint()
        fn = self.lib.nvmlDeviceGetMaxClockInfo if maximum else self.lib.nvmlDeviceGetClockInfo
        if fn(self.h, 1, self.ct.byref(v)) != 0:  # NVML_CLOCK_SM
            raise RuntimeError("nvml clock query failed")
        return int(v.value)

    def reasons(self) -> int:
        v = self.ct.c_ulonglong()
        if self.reason_fn(self.h, self.ct.byref(v)) != 0:
            raise RuntimeError("nvml clock-event query failed")
        return int(v.value)


class ClockSampler:
    """Samples the SM clock and clock-event reasons of this process's GPU (NVML through ctypes,
    located by PCI bus id; nvidia-smi as a fallback) while the timed region runs."""

    REASONS = {"hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
               "hw_power_brake": 0x80, "sw_power_cap": 0x4}

    def __init__(self, cuda_index: int, period_s: float = 0.02):
        self.cuda_index, self.period = cuda_index, period_s
        self.samples, self.reasons = [], set()
        self.max_mhz, self.error = None, None
        self.t0 = self.t1 = time.time()
        self._active = False
        self._stop = threading.Event()
        self._t = None

    def __enter__(self):
        try:
            self._nv = _Nvml(self._bus_id())
            self.max_mhz = self._nv.sm_clock(maximum=True)
        except Exception as e:  # noqa: BLE001
            return self._start_smi(f"nvml unavailable ({e.__class__.__name__}: {e})")
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        return self

    def _bus_id(self) -> str:
        import torch
        pr = torch.cuda.get_device_properties(self.cuda_index)
        return f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"

    def _start_smi(self, why: str):
        """Fallback: nvidia-smi sampling every 100 ms in a child process."""
        self.error = why + "; sampled with nvidia-smi"
        q = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.hw_power_brake_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self._smi = subprocess.Popen(["nvidia-smi", "-i", self._bus_id(), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception as e:  # noqa: BLE001
            self.error = f"{why}; nvidia-smi failed ({e!r})"
            self._smi = None
        return self

    def _run(self):
        while not self._stop.is_set():
            try:
                mhz, r = self._nv.sm_clock(), self._nv.reasons()
                if self._active:  # inside the timed region
                    self.samples.append(mhz)
                    self.reasons.update(k for k, bit in self.REASONS.items() if r & bit)
            except Exception as e:  # noqa: BLE001
                self.error = f"nvml sample: {e!r}"
            time.sleep(self.period)

    def mark(self, begin: bool):
        """Wall-clock bounds of the timed region (samples outside them are dropped)."""
        if begin:
            self.t0 = time.time()
            self._active = True
        else:
            self._active = False
            self.t1 = time.time()

    def __exit__(self, *exc):
        self._stop.set()
        if self._t:
            self._t.join()
        smi = getattr(self, "_smi", None)
        if smi is not None:
            smi.terminate()
            out, _ = smi.communicate(timeout=10)
            names = ["hw_slowdown", "sw_thermal_slowdown", "hw_thermal_slowdown", "hw_power_brake", "sw_power_cap"]
            import datetime
            for ln in out.splitlines():
                f = [x.strip() for x in ln.split(",")]
                if len(f) < 8:
                    continue
                try:
                    ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    mhz, self.max_mhz = float(f[1]), float(f[2])
                except ValueError:
                    continue
                if not (self.t0 - 0.05 <= ts <= self.t1 + 0.05):
                    continue  # keep samples taken while the timed region ran
                self.samples.append(mhz)
                self.reasons.update(n for n, v in zip(names, f[3:8]) if v.lower() == "active")

    def summary(self):
        out = {"sm_mhz": float(statistics.median(self.samples)) if self.samples else None,
               "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons), "samples": len(self.samples)}
        if self.error:
            out["error"] = self.error
        return out


# ------------------------------------------------------------------------------------ inputs
def host_inputs(cfg):
    inp = synth.scan_inputs(cfg)
    dec = synth.decode_step_inputs(cfg.replace(decode_steps=1), 0)
    return inp, dec


def to_torch(a: np.ndarray, dtype: str, device=None, pin=False):
    import torch
    if dtype == "bf16" and a.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    if pin:
        t = t.pin_memory()
    if device is not None:
        t = t.to(device)
    return t


SCAN_KEYS = ("u", "delta", "z", "B", "C")
DEC_KEYS = ("x", "delta", "z", "B", "C")


# ------------------------------------------------------------------------------------ our arm
def settle_clocks(run, stream, min_ms: float):
    """Untimed iterations after the warm-up steps until `min_ms` of device time has passed: a GPU
    that was idle raises its clocks over its first milliseconds of work, so a timed region of a few
    milliseconds that starts right after a handful of warm-up steps measures part of that ramp.
    run(i) enqueues iteration i.  Returns {"steps": n, "device_ms": t}."""
    import torch
    n, spent = 0, 0.0
    while spent < min_ms and n < 1000000:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(8):
            run(n)
            n += 1
        b.record(stream)
        b.synchronize()
        spent += a.elapsed_time(b)
    return {"steps": n, "device_ms": round(spent, 1)}


def run_ours(args, cfg, rank, world, local_rank):
    import torch
    import sequence_scan_selective_b300 as ms

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    inp, dec = host_inputs(cfg)
    params = {k: to_torch(inp[k], "f32", dev) for k in ("A", "D", "delta_bias")}
    # two input sets used alternately, so no step finds the previous step's inputs in L2
    sets = [{k: to_torch(inp[k], cfg.dtype, dev) for k in SCAN_KEYS} for _ in range(2)]
    dsets = {k: to_torch(dec[k], cfg.dtype, dev) for k in DEC_KEYS}
    y = torch.empty_like(sets[0]["u"])
    state = torch.empty((cfg.batch, cfg.dim, cfg.dstate), device=dev, dtype=torch.float32)
    ydec = torch.empty((cfg.batch, cfg.dim), device=dev, dtype=sets[0]["u"].dtype)
    stream = torch.cuda.current_stream()
    # the public API's prepared form: arguments are checked once, each launch is one C call
    if args.conv:
        cp = {k: to_torch(v, "f32", dev) for k, v in synth.conv_params(cfg, args.conv).items()}
        scans = [ms.prepare_scan_fwd_conv(s["u"], cp["conv_w"], cp["conv_bias"], s["delta"], params["A"], s["B"],
                                          s["C"], params["D"], s["z"], params["delta_bias"], True, disc=args.disc,
                                          y=y, last_state=state)[0] for s in sets]
    elif args.disc != "simple":
        scans = [ms.prepare_scan_fwd(s["u"], s["delta"], params["A"], s["B"], s["C"], params["D"], s["z"],
                                     params["delta_bias"], True, y=y, last_state=state, disc=args.disc)[0]
                 for s in sets]
    else:
        scans = [ms.prepare_scan_fwd(s["u"], s["delta"], params["A"], s["B"], s["C"], params["D"], s["z"],
                                     params["delta_bias"], True, y=y, last_state=state)[0] for s in sets]
    decode = ms.prepare_state_step(state, dsets["x"], dsets["delta"], params["A"], dsets["B"], dsets["C"],
                                   params["D"], dsets["z"], params["delta_bias"], True, y=ydec, disc=args.disc)[0]

    def step(i, ev=None):
        if ev is not None:
            ev[0].record(stream)
        scans[i % 2]()
        if ev is not None:
            ev[1].record(stream)
        decode()

    W = max(args.warmup, 3)
    for i in range(W):
        step(i)
    settle = settle_clocks(lambda i: step(W + i), stream, args.settle_ms)
    torch.cuda.synchronize()
    ms.device_status()

    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    n0 = ms.launch_count()
    with ClockSampler(local_rank) as clk:
        clk.mark(True)
        t_start.record(stream)
        for i in range(K):
            step(i, evs[i])
        t_end.record(stream)
        torch.cuda.synchronize()
        clk.mark(False)
    launches = ms.launch_count() - n0
    if dist:
        dist.barrier()
    ms.device_status()
    total_ms = t_start.elapsed_time(t_end)
    scan_avg_ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    total_ms, scan_avg_ms, launches = aggregate_ranks(dist, dev, total_ms, scan_avg_ms, launches)

    elems_step = cfg.batch * cfg.dim * (cfg.seqlen + 1)
    value = whole_job_rate(elems_step, K, world, total_ms)
    e2e = None if (args.no_e2e or args.conv or args.disc != "simple") else run_e2e(args, cfg, inp, dec, params, dev,
                                                                                  world, dist)

    peaks, kind = measured_peaks()
    sb = scan_bytes(cfg)
    achieved = sb / (scan_avg_ms * 1e-3) / 1e9
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    plain = not args.conv and args.disc == "simple"  # the committed ncu records are of the default kernel mode
    kname = fwd_kernel_name(args, cfg, torch.cuda.get_device_properties(dev).multi_processor_count)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": ncu_traffic(args.workload, kname.replace("_kernel", "")) if plain else None,
                "peak_source": f"{kind} hbm_gbs", "kernel": kname,
                "algorithmic_bytes_per_launch": sb, "kernel_avg_us": round(scan_avg_ms * 1e3, 2)}
    line = {
        "metric": METRIC, "value": value, "unit": "elements/s", "n_gpus": world, "steps": K, "warmup": W,
        "clock_settle": settle, "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded, recipe of the workload)",
        "config": {"workload": WORKLOADS[args.workload], "batch": cfg.batch, "d_inner": cfg.dim,
                   "d_state": cfg.dstate, "seq_len": cfg.seqlen, "storage": cfg.dtype,
                   "step": "fwd scan (last_state) + 1 decode step from it"
                           + (f"; causal conv (width {args.conv}) fused in front of the scan" if args.conv else "")
                           + ("; exact zero-order hold" if args.disc == "zoh" else ""),
                   "elements_per_step": elems_step, "parallelism": f"replicas x{world}",
                   "scan_kernel": kname,
                   "l2": "inputs larger than L2; two input sets alternate"},
        "roofline": roofline,
        "alu_context": alu_context(cfg, scan_avg_ms),
        "clocks": clk.summary(),
        "gpu_launches": launches,
        "e2e": e2e,
    }
    if not args.no_long and plain and args.workload in ("b14", "m130"):
        del sets, scans
        line["long_sequence"] = long_sequence_rate(dev, local_rank, cfg, scan_avg_ms, peak, kind)
    if rank == 0 and not args.no_cpu_baseline and not args.conv and args.disc == "simple":
        line["cpu_baseline"] = cpu_baseline(cfg, inp, dec)
    if dist:
        dist.destroy_process_group()
    return line


def long_sequence_rate(dev, local_rank, main_cfg, main_scan_ms, peak, peak_kind, steps=3, warmup=2):
    """The million-token scan (batch 1, d_inner 1536, N 16, L 2^20, fp32) through the same
    prepared entry point: inputs generated block by block straight into device memory (25.9 GB of
    algorithmic traffic per scan, far beyond L2), `warmup` untimed scans, then `steps` scans timed
    one by one with CUDA events on the launching stream.  Its per-element rate is reported next to
    the main workload's scan rate (elements b*d*L per second of the scan launch alone)."""
    import torch
    import sequence_scan_selective_b300 as ms

    cfg = synth.CONFIGS["long"]
    n, L = cfg.batch * cfg.dim, cfg.seqlen
    d = {k: torch.empty((cfg.batch, cfg.dim, L), device=dev, dtype=torch.float32) for k in ("u", "delta", "z")}
    for lo in range(0, n, 64):
        hi = min(n, lo + 64)
        r = synth.scan_rows(cfg, range(lo, hi))
        for k in ("u", "delta", "z"):
            d[k].view(n, L)[lo:hi].copy_(torch.from_numpy(r[k]))
    for k, v in synth.scan_bc(cfg).items():
        d[k] = to_torch(v, "f32", dev)
    p = {k: to_torch(v, "f32", dev) for k, v in synth.params(cfg).items()}
    call, y, st = ms.prepare_scan_fwd(d["u"], d["delta"], p["A"], d["B"], d["C"], p["D"], d["z"], p["delta_bias"],
                                      True)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    ms.device_status()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    n0 = ms.launch_count()
    with ClockSampler(local_rank) as clk:
        clk.mark(True)
        for a, b in evs:
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize()
        clk.mark(False)
    launches = ms.launch_count() - n0
    ms.device_status()
    avg_ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    rate = n * L / (avg_ms * 1e-3)
    main_rate = main_cfg.batch * main_cfg.dim * main_cfg.seqlen / (main_scan_ms * 1e-3)
    gbs = scan_bytes(cfg) / (avg_ms * 1e-3) / 1e9
    del d, y, st, call
    torch.cuda.empty_cache()
    return {"workload": WORKLOADS["long"].replace("scan+decode", "scan"), "steps": steps, "warmup": warmup,
            "ms_per_scan": avg_ms, "elements_per_s": rate, "main_scan_elements_per_s": main_rate,
            "ratio_to_main_scan_rate": rate / main_rate, "launches_per_scan": launches / steps,
            "algorithmic_GBps": round(gbs, 1), "frac_of_hbm": round(gbs / peak, 4),
            "peak_source": f"{peak_kind} hbm_gbs", "clocks": clk.summary()}


def fwd_kernel_name(args, cfg, nsm: int = 148) -> str:
    """The forward kernel the library picks for this run: for N <= 16 the channel-per-lane kernel
    when its 32-channel units fill the SM sub-partitions at least as well as the 8-channel units of
    the four-lanes-per-channel kernel (the library's own rule), unless --kernel says otherwise."""
    if cfg.dstate > 16 or args.kernel == "warp":
        return "scan_fwd_kernel"
    if args.kernel == "lane":
        return "scan_fwd_cl_kernel"
    slots = 4 * nsm
    lane_units = cfg.batch * (-(-cfg.dim // 32))
    if lane_units * 2 <= slots:
        return "scan_fwd_cl_kernel"
    warp_units = cfg.batch * (-(-cfg.dim // 8))
    fill = lambda u: u / (slots * -(-u // slots))
    return "scan_fwd_cl_kernel" if 1.07 * fill(lane_units) >= fill(warp_units) else "scan_fwd_kernel"


def aggregate_ranks(dist, device, total_ms: float, scan_avg_ms: float, launches: int):
    """Whole-job view of a timed region run by every rank on its own replica: the slowest rank's
    times (max over ranks) and the kernel launches of all ranks (sum).  `dist` is None for one
    process; any backend works (NCCL tensors on the GPU, gloo on the CPU)."""
    if dist is None:
        return total_ms, scan_avg_ms, launches
    import torch
    t = torch.tensor([total_ms, scan_avg_ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    lt = torch.tensor([launches], device=device, dtype=torch.float64)
    dist.all_reduce(lt)
    return float(t[0]), float(t[1]), int(lt.item())


def whole_job_rate(elems_per_step: int, steps: int, world: int, total_ms: float) -> float:
    """Elements per second of all ranks together: each rank processed elems_per_step * steps
    elements of its own replica within the (max over ranks) timed region."""
    return elems_per_step * steps * world / (total_ms * 1e-3)


def run_e2e(args, cfg, inp, dec, params, dev, world, dist):
    """Public API with host buffers: pinned host -> device copies of the step's inputs, the scan and
    the decode step, device -> host copy of both outputs, all inside the timed region.  The scan goes
    through mamba_scan_fwd_pipelined, which overlaps the copies of one batch row with the scan of
    the previous one."""
    import torch
    import sequence_scan_selective_b300 as ms

    host = {k: to_torch(inp[k], cfg.dtype, pin=True) for k in SCAN_KEYS}
    hdec = {k: to_torch(dec[k], cfg.dtype, pin=True) for k in DEC_KEYS}
    dd = {k: torch.empty_like(v, device=dev) for k, v in hdec.items()}
    ydec = torch.empty_like(dd["x"])
    state = torch.empty((cfg.batch, cfg.dim, cfg.dstate), device=dev)
    y_host = torch.empty_like(host["u"]).pin_memory()
    ydec_host = torch.empty_like(hdec["x"]).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in list(host.values()) + list(hdec.values()))
    d2h = y_host.numel() * y_host.element_size() + ydec_host.numel() * ydec_host.element_size()

    def step():
        # the scan of host-resident inputs: batch rows pipelined over copy-in, scan and copy-out
        ms.mamba_scan_fwd_pipelined(host["u"], host["delta"], params["A"], host["B"], host["C"], params["D"],
                                    host["z"], params["delta_bias"], True, y=y_host, last_state=state)
        for k in DEC_KEYS:
            dd[k].copy_(hdec[k], non_blocking=True)
        ms.mamba_state_step(state, dd["x"], dd["delta"], params["A"], dd["B"], dd["C"], params["D"], dd["z"],
                            params["delta_bias"], True, y=ydec)
        ydec_host.copy_(ydec, non_blocking=True)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    K = max(1, args.e2e_steps)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    a.record()
    for _ in range(K):
        step()
    b.record()
    torch.cuda.synchronize()
    ms_tot = a.elapsed_time(b)
    if dist:
        t = torch.tensor([ms_tot], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_tot = float(t[0])
    elems = cfg.batch * cfg.dim * (cfg.seqlen + 1) * K * world
    # context: the same bytes moved by plain copies alone (host -> device and device -> host on two
    # streams at once), the floor the host link sets for this step
    src_h = torch.empty(h2d, dtype=torch.uint8).pin_memory()
    dst_d = torch.empty(h2d, dtype=torch.uint8, device=dev)
    src_d = torch.empty(d2h, dtype=torch.uint8, device=dev)
    dst_h = torch.empty(d2h, dtype=torch.uint8).pin_memory()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    cur = torch.cuda.current_stream(dev)

    def copies():
        s_in.wait_stream(cur)
        s_out.wait_stream(cur)
        with torch.cuda.stream(s_in):
            dst_d.copy_(src_h, non_blocking=True)
        with torch.cuda.stream(s_out):
            dst_h.copy_(src_d, non_blocking=True)
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)

    copies()
    torch.cuda.synchronize()
    a.record()
    for _ in range(K):
        copies()
    b.record()
    torch.cuda.synchronize()
    link_ms = a.elapsed_time(b) / K
    return {"value": elems / (ms_tot * 1e-3), "unit": "elements/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": K, "ms_per_step": ms_tot / K,
            "copies_alone_ms_per_step": round(link_ms, 3), "copies_alone_fraction": round(link_ms / (ms_tot / K), 3)}


# ------------------------------------------------------------------------------------ CPU oracle
def _oracle_step(cfg, inp, dec, rows, nthreads):
    import oracle
    L = cfg.seqlen
    flat = {k: inp[k].reshape(cfg.batch * cfg.dim, L)[rows] for k in ("u", "delta", "z")}
    _, st = oracle.scan_rows(rows, cfg.dim, flat["u"], flat["delta"], flat["z"], inp["A"], inp["D"],
                             inp["delta_bias"], inp["B"], inp["C"], True, cfg.dtype, nthreads=nthreads)
    rb, rd = rows // cfg.dim, rows % cfg.dim
    oracle.state_step_rows(rows, cfg.dim, st, dec["x"][rb, rd], dec["delta"][rb, rd], dec["z"][rb, rd], inp["A"],
                           inp["D"], inp["delta_bias"], dec["B"], dec["C"], True, cfg.dtype, nthreads=nthreads)


def _sample_rows(cfg, budget_rows):
    n = cfg.batch * cfg.dim
    k = int(max(1, min(n, budget_rows)))
    return np.unique(np.linspace(0, n - 1, k).astype(np.int64))


def _oracle_rate(cfg, inp, dec, nthreads):
    """Channels per second of the oracle on all host threads, from a probe of several channels per
    thread (so the probe itself runs in parallel like the timed sample)."""
    _oracle_step(cfg, inp, dec, _sample_rows(cfg, nthreads), nthreads)  # warm-up: library load, threads
    probe = _sample_rows(cfg, max(16 * nthreads, 64))
    t = time.perf_counter()
    _oracle_step(cfg, inp, dec, probe, nthreads)
    return len(probe) / max(time.perf_counter() - t, 1e-4)


def cpu_baseline(cfg, inp, dec, target_s=15.0):
    """The fp64 oracle as it stands, on the host cores, over a bounded sample of the workload
    (evenly spaced channels, full sequence length each; repeated passes when the whole workload
    takes less than the target time)."""
    nthreads = os.cpu_count() or 1
    rate = _oracle_rate(cfg, inp, dec, nthreads)
    n = cfg.batch * cfg.dim
    rows = _sample_rows(cfg, target_s * rate)
    passes, t = 0, time.perf_counter()
    while True:  # passes until the target wall time (the probe's rate is only an estimate)
        _oracle_step(cfg, inp, dec, rows, nthreads)
        passes += 1
        dt = time.perf_counter() - t
        if dt >= target_s or passes >= 200:
            break
    return {"value": passes * len(rows) * (cfg.seqlen + 1) / dt, "unit": "elements/s", "cores": nthreads,
            "kind": "oracle",
            "sample": f"{passes} pass(es) over {len(rows)} of {n} channels (evenly spaced), "
                      f"full L={cfg.seqlen} scan + 1 decode step each, {dt:.1f} s wall on {nthreads} threads"}


def run_reference(args, cfg, rank):
    """Reference arm: the fp64 CPU oracle on the host cores, same metric and workload; each step is
    a bounded sample of the workload's channels so the whole run ends within a few minutes."""
    if rank != 0:
        return None
    inp, dec = host_inputs(cfg)
    nthreads = os.cpu_count() or 1
    K, W = max(1, args.steps), max(0, args.warmup)
    rate = _oracle_rate(cfg, inp, dec, nthreads)
    rows = _sample_rows(cfg, max(1.0, (120.0 / (K + W)) * rate))
    for _ in range(W):
        _oracle_step(cfg, inp, dec, rows, nthreads)
    t = time.perf_counter()
    for _ in range(K):
        _oracle_step(cfg, inp, dec, rows, nthreads)
    dt = time.perf_counter() - t
    value = len(rows) * (cfg.seqlen + 1) * K / dt
    sample = f"{len(rows)} of {cfg.batch * cfg.dim} channels per step, full L={cfg.seqlen} scan + 1 decode step"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "elements/s", "n_gpus": args.gpus,
        "steps": K, "warmup": W, "ms_per_step": dt / K * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, recipe of the workload)",
        "config": {"workload": WORKLOADS.get(args.workload, cfg.name), "batch": cfg.batch, "d_inner": cfg.dim,
                   "d_state": cfg.dstate, "seq_len": cfg.seqlen, "storage": cfg.dtype},
        "cpu_baseline": {"value": value, "unit": "elements/s", "cores": nthreads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "elements/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def _reference_line(args, cfg, value, K, W, dt, nthreads, sample, workload):
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "elements/s", "n_gpus": args.gpus,
        "steps": K, "warmup": W, "ms_per_step": dt / K * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, recipe of the workload)",
        "config": {"workload": workload, "batch": cfg.batch, "d_inner": cfg.dim, "d_state": cfg.dstate,
                   "seq_len": cfg.seqlen, "storage": cfg.dtype},
        "cpu_baseline": {"value": value, "unit": "elements/s", "cores": nthreads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "elements/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference_bwd(args, cfg, rank):
    """Reference arm of the backward pass: the oracle's gradients on a bounded, evenly spaced
    sample of channels (full L each), per step."""
    if rank != 0:
        return None
    import oracle
    nthreads = os.cpu_count() or 1
    K, W = max(1, args.steps), max(0, args.warmup)
    p = synth.params(cfg)
    bc = synth.scan_bc(cfg)
    L, N = cfg.seqlen, cfg.dstate

    def step(rows):
        x = synth.scan_rows(cfg, rows)
        dy = synth.widen(synth.grad_rows(cfg, rows), cfg.dtype)
        t = time.perf_counter()
        oracle.scan_bwd_rows(rows, cfg.batch, cfg.dim, x["u"], x["delta"], x["z"], p["A"], p["D"],
                             p["delta_bias"], bc["B"], bc["C"], dy, True, cfg.dtype,
                             synth.state_rows(cfg, rows, "h0").astype(np.float64),
                             synth.state_rows(cfg, rows, "dlast").astype(np.float64), nthreads=nthreads)
        return time.perf_counter() - t

    probe = _sample_rows(cfg, max(4 * nthreads, 16))
    rate = len(probe) / max(step(probe), 1e-4)
    rows = _sample_rows(cfg, max(1.0, (60.0 / (K + W)) * rate))
    for _ in range(W):
        step(rows)
    dt = sum(step(rows) for _ in range(K))  # oracle time only (input generation excluded)
    value = len(rows) * L * K / dt
    sample = f"{len(rows)} of {cfg.batch * cfg.dim} channels per step, full L={L} backward pass"
    return _reference_line(args, cfg, value, K, W, dt, nthreads, sample,
                           WORKLOADS[args.workload].replace("scan+decode", "backward pass"))


def run_reference_decode(args, cfg, rank):
    """Reference arm of the decode workload: the oracle's decode step over a bounded sample of
    channels, fresh inputs per step."""
    if rank != 0:
        return None
    import oracle
    nthreads = os.cpu_count() or 1
    K, W = max(1, args.steps), max(0, args.warmup)
    p = synth.params(cfg)
    bsz = cfg.batch
    n = bsz * cfg.dim
    rows = _sample_rows(cfg, min(n, 65536))
    rb, rd = rows // cfg.dim, rows % cfg.dim
    state = synth.decode_state0(cfg).reshape(n, cfg.dstate)[rows].astype(np.float64)
    steps = [synth.decode_step_inputs(cfg, s) for s in range(min(K + W, 8))]
    dt = 0.0
    for i in range(K + W):
        s = steps[i % len(steps)]
        t = time.perf_counter()
        oracle.state_step_rows(rows, cfg.dim, state, s["x"][rb, rd], s["delta"][rb, rd], s["z"][rb, rd], p["A"],
                               p["D"], p["delta_bias"], s["B"], s["C"], True, cfg.dtype, nthreads=nthreads)
        if i >= W:
            dt += time.perf_counter() - t
    value = len(rows) * K / dt
    sample = f"{len(rows)} of {n} channels per step, {K} steps"
    return _reference_line(args, cfg, value, K, W, dt, nthreads, sample, WORKLOADS["decode"])


def run_decode(args, cfg, rank, world, local_rank):
    """Consecutive decode steps (mamba_state_step) on the decode workload, each step with fresh
    x, delta, z, B, C: timed as one block of plain launches and, separately, as the same steps
    captured in one CUDA graph and replayed.  The fp32 state (41.9 MB at this shape) stays in the
    126 MB L2 between steps, so the step can run above the HBM rate; `traffic` is then the DRAM
    share that actually moves."""
    import torch
    import sequence_scan_selective_b300 as ms

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    S = max(1, min(args.steps, args.decode_inputs))  # distinct pre-generated steps, cycled
    dec = synth.decode_inputs(cfg, S)
    p = {k: to_torch(v, "f32", dev) for k, v in synth.params(cfg).items()}
    d = {k: to_torch(dec[k], cfg.dtype, dev) for k in DEC_KEYS}
    state = to_torch(synth.decode_state0(cfg), "f32", dev)
    y = torch.empty((S, cfg.batch, cfg.dim), device=dev, dtype=d["x"].dtype)
    calls = [ms.prepare_state_step(state, d["x"][i], d["delta"][i], p["A"], d["B"][i], d["C"][i], p["D"],
                                   d["z"][i], p["delta_bias"], True, y=y[i])[0] for i in range(S)]
    stream = torch.cuda.current_stream()
    W = max(args.warmup, 3)
    for i in range(W):
        calls[i % S]()
    settle = settle_clocks(lambda i: calls[(W + i) % S](), stream, args.settle_ms)
    torch.cuda.synchronize()
    K = args.steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    n0 = ms.launch_count()
    with ClockSampler(local_rank) as clk:
        clk.mark(True)
        ev[0].record(stream)
        for i in range(K):
            calls[i % S]()
        ev[1].record(stream)
        torch.cuda.synchronize()
        clk.mark(False)
    launches = ms.launch_count() - n0
    total_ms = ev[0].elapsed_time(ev[1])
    # the same S steps as one CUDA graph (captured on a side stream, replayed on this one)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        gcalls = [ms.prepare_state_step(state, d["x"][i], d["delta"][i], p["A"], d["B"][i], d["C"][i], p["D"],
                                        d["z"][i], p["delta_bias"], True, y=y[i])[0] for i in range(S)]
        with torch.cuda.graph(graph, stream=side):
            for c in gcalls:
                c()
    stream.wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    reps = max(1, K // S)
    ev[2].record(stream)
    for _ in range(reps):
        graph.replay()
    ev[3].record(stream)
    torch.cuda.synchronize()
    graph_ms = ev[2].elapsed_time(ev[3]) / (reps * S)
    # the same steps on R state buffers used in turn (R independent decode streams, each step
    # still one launch over the whole batch): the states total more than twice the L2, so every
    # step streams its state from HBM and back
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    sbytes = state.numel() * 4
    R = max(args.decode_states, -(-2 * l2 // sbytes) + 1)
    rstates = [state.clone() for _ in range(R)]
    rcalls = [ms.prepare_state_step(rstates[r], d["x"][i], d["delta"][i], p["A"], d["B"][i], d["C"][i], p["D"],
                                    d["z"][i], p["delta_bias"], True, y=y[i])[0]
              for r in range(R) for i in range(min(S, 8))]
    nrc = len(rcalls)
    for i in range(2 * R):
        rcalls[i % nrc]()
    torch.cuda.synchronize()
    ev2 = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev2[0].record(stream)
    for i in range(K):  # step i uses state buffer i % R
        rcalls[(i % R) * min(S, 8) + (i // R) % min(S, 8)]()
    ev2[1].record(stream)
    torch.cuda.synchronize()
    rot_ms = ev2[0].elapsed_time(ev2[1]) / K
    del rstates, rcalls
    total_ms, avg_ms, launches = aggregate_ranks(dist, dev, total_ms, total_ms / K, launches)
    elems_step = cfg.batch * cfg.dim
    peaks, kind = measured_peaks()
    sb = step_bytes(cfg)
    achieved = sb / (avg_ms * 1e-3) / 1e9
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    line = {
        "metric": METRIC, "value": whole_job_rate(elems_step, K, world, total_ms), "unit": "elements/s",
        "n_gpus": world, "steps": K, "warmup": W, "clock_settle": settle, "ms_per_step": total_ms / K,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded, recipe of the workload)",
        "config": {"workload": WORKLOADS["decode"], "batch": cfg.batch, "d_inner": cfg.dim, "d_state": cfg.dstate,
                   "storage": cfg.dtype, "step": "one decode step (state update in place), fresh inputs per step",
                   "elements_per_step": elems_step, "distinct_step_inputs": S, "parallelism": f"replicas x{world}",
                   "l2": "state L2-resident between steps (41.9 MB); step inputs cycle through S distinct sets"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": ncu_traffic("decode", "state_step") if args.disc == "simple" else None,
                     "peak_source": f"{kind} hbm_gbs",
                     "kernel": "state_step_kernel", "algorithmic_bytes_per_launch": sb,
                     "kernel_avg_us": round(avg_ms * 1e3, 3)},
        "graph": {"us_per_step": round(graph_ms * 1e3, 3), "steps_per_graph": S,
                  "elements_per_s": elems_step * world / (graph_ms * 1e-3)},
        "rotating_states": {"state_buffers": R, "state_bytes_total": R * sbytes, "l2_bytes": l2,
                            "us_per_step": round(rot_ms * 1e3, 3),
                            "elements_per_s": elems_step * world / (rot_ms * 1e-3),
                            "achieved_GBps": round(sb / (rot_ms * 1e-3) / 1e9, 1),
                            "frac_of_hbm": round(sb / (rot_ms * 1e-3) / 1e9 / peak, 4)},
        "clocks": clk.summary(),
        "gpu_launches": launches,
        "e2e": None,
    }
    if dist:
        dist.destroy_process_group()
    return line


def run_bwd(args, cfg, rank, world, local_rank):
    """The backward pass alone (mamba_scan_bwd: recompute + reverse sweep), device-timed."""
    import torch
    import sequence_scan_selective_b300 as ms

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    inp = synth.scan_inputs(cfg)
    g = synth.grad_inputs(cfg)
    params = {k: to_torch(inp[k], "f32", dev) for k in ("A", "D", "delta_bias")}
    sets = []
    for _ in range(2):  # two input sets used alternately (inputs larger than L2)
        st = {k: to_torch(inp[k], cfg.dtype, dev) for k in SCAN_KEYS}
        st["dy"] = to_torch(g["dy"], cfg.dtype, dev)
        st["h0"] = to_torch(g["h0"], "f32", dev)
        st["dlast"] = to_torch(g["dlast"], "f32", dev)
        sets.append(st)
    out = None
    calls = []
    if args.conv:  # the block's backward pass: convolution recomputed, scan gradients, convolution gradients
        cp = {k: to_torch(v, "f32", dev) for k, v in synth.conv_params(cfg, args.conv).items()}
        for st in sets:
            calls.append(lambda st=st: ms.mamba_scan_bwd_conv(
                st["u"], cp["conv_w"], cp["conv_bias"], st["delta"], params["A"], st["B"], st["C"], st["dy"],
                params["D"], st["z"], params["delta_bias"], True, h0=st["h0"], dlast_state=st["dlast"]))
    else:
        for st in sets:
            c, out = ms.prepare_scan_bwd(st["u"], st["delta"], params["A"], st["B"], st["C"], st["dy"],
                                         params["D"], st["z"], params["delta_bias"], True, h0=st["h0"],
                                         dlast_state=st["dlast"], out=out)
            calls.append(c)
    stream = torch.cuda.current_stream()
    W = max(args.warmup, 3)
    for i in range(W):
        calls[i % 2]()
    settle = settle_clocks(lambda i: calls[(W + i) % 2](), stream, args.settle_ms)
    torch.cuda.synchronize()
    K = args.steps
    # events around each call as well: the kernel time excludes any gap the host leaves between calls
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    n0 = ms.launch_count()
    with ClockSampler(local_rank) as clk:
        clk.mark(True)
        t_start.record(stream)
        for i in range(K):
            evs[i][0].record(stream)
            calls[i % 2]()
            evs[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        clk.mark(False)
    launches = ms.launch_count() - n0
    total_ms = t_start.elapsed_time(t_end)
    call_ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    total_ms, avg_ms, launches = aggregate_ranks(dist, dev, total_ms, call_ms, launches)
    train = None
    if not args.conv and cfg.dstate <= 16:
        train = train_step_times(ms, sets, params, out, stream, W, K)
    elems_step = cfg.batch * cfg.dim * cfg.seqlen
    peaks, kind = measured_peaks()
    bb = bwd_bytes(cfg)
    if args.conv:  # x read twice, u written and read back by the scan, du read: 4 more element passes
        bb += 4 * cfg.batch * cfg.dim * cfg.seqlen * (2 if cfg.dtype == "bf16" else 4)
    achieved = bb / (avg_ms * 1e-3) / 1e9
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    line = {
        "metric": METRIC, "value": whole_job_rate(elems_step, K, world, total_ms), "unit": "elements/s",
        "n_gpus": world, "steps": K, "warmup": W, "clock_settle": settle, "ms_per_step": total_ms / K,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded, recipe of the workload)",
        "config": {"workload": WORKLOADS[args.workload].replace("scan+decode", "backward pass"),
                   "batch": cfg.batch, "d_inner": cfg.dim, "d_state": cfg.dstate, "seq_len": cfg.seqlen,
                   "storage": cfg.dtype,
                   "step": (f"backward pass of the causal convolution (width {args.conv}) and the scan: gradients "
                            "of x, conv weights and bias, delta, z, A, B, C, D, bias, h0" if args.conv else
                            "backward pass: gradients of u, delta, z, A, B, C, D, bias, h0"),
                   "elements_per_step": elems_step, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2; two input sets alternate"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": None if args.conv else ncu_traffic(args.workload, "scan_bwd"),
                     "peak_source": f"{kind} hbm_gbs",
                     "kernel": "conv_fwd + scan_bwd + conv_bwd" if args.conv else "scan_bwd_kernel",
                     "algorithmic_bytes_per_launch": bb,
                     "kernel_avg_us": round(avg_ms * 1e3, 2)},
        "clocks": clk.summary(),
        "gpu_launches": launches,
        "e2e": None,
    }
    if train is not None:
        line["train_step"] = train
    if dist:
        dist.destroy_process_group()
    return line


def train_step_times(ms, sets, params, out, stream, W, K):
    """Forward + backward of one training step, two ways: the forward scan and a backward pass that
    recomputes its checkpoints in a forward sweep, or the training forward pass (which writes the
    checkpoints) and a backward pass that starts from them.  Each leg device-timed alone over K
    launches, the input sets alternating as in the backward line."""
    import torch

    ys = [torch.empty_like(st["u"]) for st in sets]
    lss = [torch.empty_like(st["h0"]) for st in sets]
    cks = [torch.empty((st["u"].shape[0], (st["u"].shape[2] + 7) // 8, st["u"].shape[1], 16),
                       device=st["u"].device, dtype=torch.float32) for st in sets]
    got = [None, None]

    def fwd(i):
        st = sets[i]
        ms.mamba_scan_fwd(st["u"], st["delta"], params["A"], st["B"], st["C"], params["D"], st["z"],
                          params["delta_bias"], True, y=ys[i], last_state=lss[i], h0=st["h0"])

    def fwd_train(i):
        st = sets[i]
        _, _, got[i] = ms.mamba_scan_fwd_train(st["u"], st["delta"], params["A"], st["B"], st["C"], params["D"],
                                               st["z"], params["delta_bias"], True, h0=st["h0"], y=ys[i],
                                               last_state=lss[i], ckpt=cks[i])

    for i in range(2):
        fwd_train(i)
    torch.cuda.synchronize()
    if got[0] is None:  # the planner split the forward pass: no checkpoints for this shape
        return {"checkpoints": "not kept (the forward pass splits the sequence for this shape)"}
    bwd_ck = []
    for i, st in enumerate(sets):
        c, _ = ms.prepare_scan_bwd(st["u"], st["delta"], params["A"], st["B"], st["C"], st["dy"], params["D"],
                                   st["z"], params["delta_bias"], True, h0=st["h0"], dlast_state=st["dlast"],
                                   out=out, ckpt=cks[i])
        bwd_ck.append(c)
    bwd_plain = []
    for st in sets:
        c, _ = ms.prepare_scan_bwd(st["u"], st["delta"], params["A"], st["B"], st["C"], st["dy"], params["D"],
                                   st["z"], params["delta_bias"], True, h0=st["h0"], dlast_state=st["dlast"],
                                   out=out)
        bwd_plain.append(c)

    def timed(fn):
        for i in range(W):
            fn(i % 2)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(K):
            fn(i % 2)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / K * 1e3

    us = {"fwd": timed(fwd), "bwd": timed(lambda i: bwd_plain[i]()),
          "fwd_train": timed(fwd_train), "bwd_from_checkpoints": timed(lambda i: bwd_ck[i]())}
    plain, ck = us["fwd"] + us["bwd"], us["fwd_train"] + us["bwd_from_checkpoints"]
    return {"us": {k: round(v, 2) for k, v in us.items()},
            "recompute_us": round(plain, 2), "checkpoints_us": round(ck, 2), "speedup": round(plain / ck, 4),
            "note": "forward + backward of one step; checkpoints: the training forward pass writes the state "
                    "before every 8-step slot and the backward pass skips its forward sweep"}


def main():
    args = parse()
    if args.kernel != "auto":
        os.environ["MAMBA_SCAN_KERNEL"] = args.kernel
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = synth.CONFIGS[args.workload]
    if args.seqlen > 0 and args.workload != "decode":
        cfg = cfg.replace(seqlen=args.seqlen)
        WORKLOADS[args.workload] = WORKLOADS[args.workload].replace(
            f"L {synth.CONFIGS[args.workload].seqlen}", f"L {args.seqlen}")
    if args.impl == "reference" and args.workload == "decode":
        line = run_reference_decode(args, cfg, rank)
    elif args.impl == "reference" and args.which == "bwd":
        line = run_reference_bwd(args, cfg, rank)
    elif args.impl == "reference":
        line = run_reference(args, cfg, rank)
    elif args.workload == "decode":
        line = run_decode(args, cfg, rank, world, local_rank)
    elif args.which == "bwd":
        line = run_bwd(args, cfg, rank, world, local_rank)
    else:
        line = run_ours(args, cfg, rank, world, local_rank)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
