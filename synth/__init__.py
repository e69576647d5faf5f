"""Seeded synthetic inputs for the selective scan and its single-token state update.

This module is shared by the tests, the benchmark and the oracle's checks.  It holds no arithmetic of
the scan itself: it only draws random tensors with the shapes and value distributions of the Mamba
layer workloads, and stores them in the number formats the scan consumes (fp32, or bf16 kept as
uint16 bit patterns).

Every random row comes from its own stream, keyed by (seed, tensor, row), so any subset of rows
(for example a few sampled channels of a million-token sequence) can be regenerated on its own and
is bit-identical to the same rows of the full tensor.

Recipe (selective-SSM layer of "Mamba: Linear-Time Sequence Modeling with Selective State Spaces",
section 3.2 of the visual guide: B, C and the step size carry batch and length dimensions, A does not):

* A[d, n] = -(n + 1)                       (real diagonal, same for every channel)
* step size Delta log-uniform in [1e-3, 0.1]; the raw input delta is chosen so that
  softplus(delta + delta_bias[d]) equals that Delta before storage rounding.  With ``bias='zero'``
  delta_bias = 0; with ``bias='loguniform'`` delta_bias[d] = softplus^-1(Delta0[d]) with Delta0
  log-uniform in the same range, and delta = softplus^-1(Delta) - delta_bias[d].
* u, z, B, C ~ N(0, 1); D = 1 (``d_mode='one'``) or D ~ N(1, 0.1) (``d_mode='normal'``).
* decode: initial state h ~ N(0, 1); each step draws fresh x, delta, z [batch, dim] and
  B, C [batch, N] with the distributions above.

softplus^-1(v) = log(expm1(v)) is used here only to place the raw inputs; the scan computes softplus.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os
from typing import Iterable, Optional, Sequence

import numpy as np

DELTA_MIN = 1e-3
DELTA_MAX = 1e-1

# tensor ids used in the stream keys
_T_U, _T_DELTA, _T_Z, _T_B, _T_C, _T_D, _T_BIAS, _T_H0 = range(1, 9)
# decode tensors use separate ids so they never share a stream with the scan tensors
_T_DX, _T_DDELTA, _T_DZ, _T_DB, _T_DC = range(11, 16)
# backward-pass inputs: gradient at y, gradient at last_state, initial state of a scan
_T_DY, _T_DLAST, _T_SH0 = range(21, 24)
# causal convolution in front of the scan: weights, bias, inputs before position 0
_T_CW, _T_CB, _T_CPREV = range(31, 34)


@dataclasses.dataclass(frozen=True)
class ScanConfig:
    """One workload: sizes, storage dtype of u/delta/z/B/C/y, and the input recipe."""

    name: str
    batch: int
    dim: int
    dstate: int
    seqlen: int
    dtype: str  # "f32" or "bf16"
    seed: int
    bias: str = "loguniform"  # "zero" or "loguniform"
    d_mode: str = "normal"  # "one" or "normal"
    softplus: bool = True
    gate: bool = True
    decode_steps: int = 0  # > 0 marks a decode workload

    @property
    def elements(self) -> int:
        return self.batch * self.dim * self.seqlen

    def replace(self, **kw) -> "ScanConfig":
        return dataclasses.replace(self, **kw)


# The five workloads.  Names say what they are; sizes follow the Mamba-130M and Mamba-1.4B layer
# shapes (d_inner 1536 / 4096, N = 16), a million-token sequence, and batched decoding.
CONFIGS = {
    "tiny": ScanConfig("tiny", 1, 16, 4, 64, "f32", seed=0, bias="zero", d_mode="one"),
    "m130": ScanConfig("m130", 8, 1536, 16, 2048, "f32", seed=1),
    "b14": ScanConfig("b14", 4, 4096, 16, 2048, "bf16", seed=2),
    "long": ScanConfig("long", 1, 1536, 16, 1 << 20, "f32", seed=3),
    "decode": ScanConfig("decode", 128, 5120, 16, 1, "bf16", seed=4, decode_steps=1000),
}


def _rng(seed: int, tensor: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor, *key])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); returns the uint16 bit patterns."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (bits + 0x7FFF + ((bits >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """Stored values as float64 (exact)."""
    if dtype == "bf16":
        return bf16_bits_to_f32(x).astype(np.float64)
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    x32 = np.asarray(x, dtype=np.float32)
    return f32_to_bf16_bits(x32) if dtype == "bf16" else x32


def _loguniform(g: np.random.Generator, n) -> np.ndarray:
    lo, hi = np.log(DELTA_MIN), np.log(DELTA_MAX)
    return np.exp(lo + g.random(n) * (hi - lo))


def _softplus_inv(v: np.ndarray) -> np.ndarray:
    return np.log(np.expm1(v))


def params(cfg: ScanConfig) -> dict:
    """Per-channel parameters: A [dim, N], D [dim], delta_bias [dim] (all fp32)."""
    A = -np.tile(np.arange(1, cfg.dstate + 1, dtype=np.float32), (cfg.dim, 1))
    if cfg.d_mode == "one":
        D = np.ones(cfg.dim, dtype=np.float32)
    else:
        D = (1.0 + 0.1 * _rng(cfg.seed, _T_D).standard_normal(cfg.dim)).astype(np.float32)
    if cfg.bias == "zero":
        bias = np.zeros(cfg.dim, dtype=np.float32)
    else:
        bias = _softplus_inv(_loguniform(_rng(cfg.seed, _T_BIAS), cfg.dim)).astype(np.float32)
    return {"A": np.ascontiguousarray(A), "D": D, "delta_bias": bias}


def _row_u(cfg, r, L):
    return _rng(cfg.seed, _T_U, r).standard_normal(L, dtype=np.float32)


def _row_z(cfg, r, L):
    return _rng(cfg.seed, _T_Z, r).standard_normal(L, dtype=np.float32)


def _row_delta(cfg, r, L, bias_d):
    dl = _loguniform(_rng(cfg.seed, _T_DELTA, r), L)
    return _softplus_inv(dl) - np.float64(bias_d)


def _workers(n: int) -> int:
    return max(1, min(n, os.cpu_count() or 1, 32))


def _fill_rows(out: np.ndarray, rows: Sequence[int], fn, dtype: str, threads: Optional[int] = None):
    """out[i, :] = store(fn(rows[i])), computed by a thread pool over row blocks."""
    n = len(rows)

    def work(lo, hi):
        for i in range(lo, hi):
            out[i] = _store(fn(int(rows[i])), dtype)

    nt = threads or _workers(n)
    if nt <= 1 or n < 4:
        work(0, n)
        return
    step = (n + nt * 4 - 1) // (nt * 4)
    with _cf.ThreadPoolExecutor(nt) as ex:
        list(ex.map(lambda lo: work(lo, min(n, lo + step)), range(0, n, step)))


def _storage_dtype(dtype: str):
    return np.uint16 if dtype == "bf16" else np.float32


def scan_bc(cfg: ScanConfig, seqlen: Optional[int] = None) -> dict:
    """B, C [batch, N, L] in the storage dtype."""
    L = seqlen or cfg.seqlen
    out = {}
    for name, tid in (("B", _T_B), ("C", _T_C)):
        arr = np.empty((cfg.batch * cfg.dstate, L), dtype=_storage_dtype(cfg.dtype))
        _fill_rows(arr, range(cfg.batch * cfg.dstate),
                   lambda r, tid=tid: _rng(cfg.seed, tid, r).standard_normal(L, dtype=np.float32), cfg.dtype)
        out[name] = arr.reshape(cfg.batch, cfg.dstate, L)
    return out


def scan_rows(cfg: ScanConfig, rows: Iterable[int], seqlen: Optional[int] = None,
              tensors: Sequence[str] = ("u", "delta", "z")) -> dict:
    """u, delta, z for the given flat channel rows r = b * dim + d, each [len(rows), L]."""
    rows = np.asarray(list(rows), dtype=np.int64)
    L = seqlen or cfg.seqlen
    p = params(cfg)
    sd = _storage_dtype(cfg.dtype)
    out = {"rows": rows}
    for name in tensors:
        arr = np.empty((len(rows), L), dtype=sd)
        if name == "u":
            fn = lambda r: _row_u(cfg, r, L)
        elif name == "z":
            fn = lambda r: _row_z(cfg, r, L)
        elif name == "delta":
            fn = lambda r: _row_delta(cfg, r, L, p["delta_bias"][r % cfg.dim])
        else:
            raise ValueError(name)
        _fill_rows(arr, rows, fn, cfg.dtype)
        out[name] = arr
    return out


def scan_inputs(cfg: ScanConfig, seqlen: Optional[int] = None) -> dict:
    """Full inputs of one forward scan: u, delta, z [batch, dim, L]; B, C [batch, N, L];
    A [dim, N]; D, delta_bias [dim].  u/delta/z/B/C are fp32 or bf16 bit patterns (uint16)."""
    L = seqlen or cfg.seqlen
    out = dict(params(cfg))
    rows = scan_rows(cfg, range(cfg.batch * cfg.dim), L)
    for k in ("u", "delta", "z"):
        out[k] = rows[k].reshape(cfg.batch, cfg.dim, L)
    out.update(scan_bc(cfg, L))
    return out


# ----------------------------------------------------------------------------------------- backward
def grad_rows(cfg: ScanConfig, rows: Iterable[int], seqlen: Optional[int] = None) -> np.ndarray:
    """Gradient arriving at y for the given flat channel rows: N(0, 1), [len(rows), L] in the
    storage dtype."""
    rows = np.asarray(list(rows), dtype=np.int64)
    L = seqlen or cfg.seqlen
    arr = np.empty((len(rows), L), dtype=_storage_dtype(cfg.dtype))
    _fill_rows(arr, rows, lambda r: _rng(cfg.seed, _T_DY, r).standard_normal(L, dtype=np.float32), cfg.dtype)
    return arr


def state_rows(cfg: ScanConfig, rows: Iterable[int], which: str) -> np.ndarray:
    """Per-channel fp32 state-shaped inputs, N(0, 1), [len(rows), N]: ``which`` = "h0" (initial
    state of a scan) or "dlast" (gradient arriving at last_state)."""
    rows = np.asarray(list(rows), dtype=np.int64)
    tid = {"h0": _T_SH0, "dlast": _T_DLAST}[which]
    arr = np.empty((len(rows), cfg.dstate), dtype=np.float32)
    _fill_rows(arr, rows, lambda r: _rng(cfg.seed, tid, r).standard_normal(cfg.dstate, dtype=np.float32),
               "f32")
    return arr


def grad_inputs(cfg: ScanConfig, seqlen: Optional[int] = None) -> dict:
    """Backward-pass inputs for the whole workload: dy [batch, dim, L] (storage dtype),
    dlast_state and h0 [batch, dim, N] (fp32)."""
    L = seqlen or cfg.seqlen
    rows = range(cfg.batch * cfg.dim)
    return {"dy": grad_rows(cfg, rows, L).reshape(cfg.batch, cfg.dim, L),
            "dlast": state_rows(cfg, rows, "dlast").reshape(cfg.batch, cfg.dim, cfg.dstate),
            "h0": state_rows(cfg, rows, "h0").reshape(cfg.batch, cfg.dim, cfg.dstate)}


# ----------------------------------------------------------------------------------------- convolution
def conv_params(cfg: ScanConfig, K: int = 4) -> dict:
    """Depthwise causal convolution of width K in front of the scan: conv_w [dim, K] and
    conv_bias [dim], uniform on [-1/sqrt(K), 1/sqrt(K)] (the fan-in scale of a depthwise
    convolution).  The scan's u tensor then serves as the convolution's input x."""
    lim = 1.0 / np.sqrt(K)
    w = _rng(cfg.seed, _T_CW, K).uniform(-lim, lim, size=(cfg.dim, K)).astype(np.float32)
    b = _rng(cfg.seed, _T_CB, K).uniform(-lim, lim, size=cfg.dim).astype(np.float32)
    return {"conv_w": w, "conv_bias": b}


def conv_prev(cfg: ScanConfig, K: int = 4) -> np.ndarray:
    """Inputs before position 0 for a convolution of width K: N(0, 1), fp32 [batch, dim, K-1]."""
    g = _rng(cfg.seed, _T_CPREV, K)
    return g.standard_normal((cfg.batch, cfg.dim, max(K - 1, 0)), dtype=np.float32)


# ----------------------------------------------------------------------------------------- decode
def decode_state0(cfg: ScanConfig, batches: Optional[Iterable[int]] = None) -> np.ndarray:
    """Initial state h ~ N(0,1), fp32 [len(batches), dim, N] (all batches by default)."""
    bs = list(range(cfg.batch)) if batches is None else list(batches)
    out = np.empty((len(bs), cfg.dim * cfg.dstate), dtype=np.float32)
    _fill_rows(out, bs, lambda b: _rng(cfg.seed, _T_H0, b).standard_normal(cfg.dim * cfg.dstate,
                                                                            dtype=np.float32), "f32")
    return out.reshape(len(bs), cfg.dim, cfg.dstate)


def decode_step_inputs(cfg: ScanConfig, step: int, batches: Optional[Iterable[int]] = None) -> dict:
    """Inputs of decode step ``step``: x, delta, z [len(batches), dim]; B, C [len(batches), N]."""
    bs = list(range(cfg.batch)) if batches is None else list(batches)
    p = params(cfg)
    sd = _storage_dtype(cfg.dtype)
    out = {}
    for name, tid in (("x", _T_DX), ("z", _T_DZ)):
        arr = np.empty((len(bs), cfg.dim), dtype=sd)
        _fill_rows(arr, bs, lambda b, tid=tid: _rng(cfg.seed, tid, step, b).standard_normal(
            cfg.dim, dtype=np.float32), cfg.dtype, threads=1)
        out[name] = arr
    arr = np.empty((len(bs), cfg.dim), dtype=sd)
    _fill_rows(arr, bs, lambda b: _softplus_inv(_loguniform(_rng(cfg.seed, _T_DDELTA, step, b), cfg.dim))
               - p["delta_bias"].astype(np.float64), cfg.dtype, threads=1)
    out["delta"] = arr
    for name, tid in (("B", _T_DB), ("C", _T_DC)):
        arr = np.empty((len(bs), cfg.dstate), dtype=sd)
        _fill_rows(arr, bs, lambda b, tid=tid: _rng(cfg.seed, tid, step, b).standard_normal(
            cfg.dstate, dtype=np.float32), cfg.dtype, threads=1)
        out[name] = arr
    return out


def decode_inputs(cfg: ScanConfig, steps: Optional[int] = None) -> dict:
    """All decode steps stacked: x, delta, z [steps, batch, dim]; B, C [steps, batch, N]."""
    S = cfg.decode_steps if steps is None else steps
    sd = _storage_dtype(cfg.dtype)
    out = {k: np.empty((S, cfg.batch, cfg.dim), dtype=sd) for k in ("x", "delta", "z")}
    out.update({k: np.empty((S, cfg.batch, cfg.dstate), dtype=sd) for k in ("B", "C")})

    def work(s):
        st = decode_step_inputs(cfg, s)
        for k, v in st.items():
            out[k][s] = v

    with _cf.ThreadPoolExecutor(_workers(S)) as ex:
        list(ex.map(work, range(S)))
    return out
