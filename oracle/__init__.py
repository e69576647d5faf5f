"""fp64 CPU oracle of the selective scan — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import this
package.  The product package never imports it, and it imports nothing from the product package.

The arithmetic lives in ``oracle.c`` (plain C, double precision, sequential in time); this module
only compiles it with gcc on first use and marshals numpy arrays into it.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests.
``tests/test_oracle_pins.py`` pins the forward scan and the decode step (LTI convolution by brute
force, the scalar-state closed form, the one-step formula, the Delta -> 0 and Delta -> infinity
limits, linearity in the input, the decode step against the scan).
``tests/test_oracle_grad_pins.py`` pins the exact zero-order hold (against a numerical solution of
the held-input ODE by scipy) and the gradients (against Richardson-extrapolated central
differences of the forward, input by input).  ``tests/test_oracle_conv_pins.py`` pins the causal
convolution (against numpy's convolve) and its gradient ``causal_conv_bwd`` (against central
differences of a numpy-convolve forward, and the full-convolution form of the input gradient).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F64 = 0, 1, 2
_DT = {"f32": F32, "bf16": BF16, "f64": F64}


_P, _I, _LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
SIGNATURES = {
    "oracle_version": [],
    "oracle_scan_rows": [_LL, _P, _P, _I, _I, _LL, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P,
                         _P, _I],
    "oracle_scan_rows_ex": [_LL, _P, _P, _I, _I, _LL, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _P,
                            _P, _P, _I],
    "oracle_state_step_rows": [_LL, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P,
                               _I],
    "oracle_state_step_rows_ex": [_LL, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I,
                                  _P, _I],
    "oracle_causal_conv_rows": [_LL, _P, _I, _I, _LL, _I, _P, _P, _P, _I, _P, _P],
    "oracle_scan_bwd_rows": [_LL, _P, _P, _I, _I, _I, _LL, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I,
                             _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I],
}
DISC = {"simple": 0, "zoh": 1}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, OpenMP, strict IEEE double arithmetic)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P, I, LL, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_double
            for name, argtypes in SIGNATURES.items():
                getattr(L, name).restype = I
                getattr(L, name).argtypes = argtypes
            _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _storage(a, dt):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype={BF16: np.uint16, F32: np.float32, F64: np.float64}[dt])


def scan_rows(rows, dim, u_rows, delta_rows, z_rows, A, D, delta_bias, B, C, softplus=True,
              dtype="f32", h0_rows=None, nthreads=0, disc="simple"):
    """Scan for the channels ``rows`` (flat b*dim + d).  u/delta/z_rows [nrows, L] in storage
    dtype; B, C [batch, N, L].  ``disc`` is "simple" (Bbar = Delta B) or "zoh" (exact zero-order
    hold).  Returns (y [nrows, L], state [nrows, N]) in float64."""
    dt = _DT[dtype]
    rows = np.asarray(rows, dtype=np.int64)
    nrows = len(rows)
    A = _c(A, np.float32)
    N = A.shape[1]
    L = np.asarray(u_rows).shape[-1]
    rb = np.ascontiguousarray(rows // dim, dtype=np.int32)
    rd = np.ascontiguousarray(rows % dim, dtype=np.int32)
    u_rows, delta_rows, z_rows = (_storage(x, dt) for x in (u_rows, delta_rows, z_rows))
    B, C = _storage(B, dt), _storage(C, dt)
    D, delta_bias = _c(D, np.float32), _c(delta_bias, np.float32)
    h0 = _c(h0_rows, np.float64)
    y = np.empty((nrows, L), dtype=np.float64)
    st = np.empty((nrows, N), dtype=np.float64)
    if disc == "simple":  # the plain entry point, so a planted mistake in it is seen by every pin
        rc = lib().oracle_scan_rows(nrows, _ptr(rb), _ptr(rd), dim, N, L, dt, _ptr(u_rows),
                                    _ptr(delta_rows), _ptr(z_rows), _ptr(A), _ptr(D),
                                    _ptr(delta_bias), _ptr(B), _ptr(C), int(bool(softplus)),
                                    _ptr(h0), _ptr(y), _ptr(st), int(nthreads))
    else:
        rc = lib().oracle_scan_rows_ex(nrows, _ptr(rb), _ptr(rd), dim, N, L, dt, _ptr(u_rows),
                                       _ptr(delta_rows), _ptr(z_rows), _ptr(A), _ptr(D),
                                       _ptr(delta_bias), _ptr(B), _ptr(C), int(bool(softplus)),
                                       DISC[disc], _ptr(h0), _ptr(y), _ptr(st), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_scan_rows rejected its arguments (rc={rc})")
    return y, st


def scan(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, dtype="f32", h0=None,
         nthreads=0, disc="simple"):
    """Full scan.  u, delta, z [batch, dim, L]; returns y [batch, dim, L], last_state [batch, dim, N]
    (float64)."""
    bsz, dim, L = np.asarray(u).shape
    N = np.asarray(A).shape[1]
    rows = np.arange(bsz * dim)
    r = lambda x: None if x is None else np.asarray(x).reshape(bsz * dim, L)
    y, st = scan_rows(rows, dim, r(u), r(delta), r(z), A, D, delta_bias, B, C, softplus, dtype,
                      None if h0 is None else np.asarray(h0, dtype=np.float64).reshape(bsz * dim, N),
                      nthreads, disc)
    return y.reshape(bsz, dim, L), st.reshape(bsz, dim, N)


def state_step_rows(rows, dim, state_rows, x_rows, delta_rows, z_rows, A, D, delta_bias, B, C,
                    softplus=True, dtype="f32", nthreads=0, disc="simple"):
    """One decode step for channels ``rows``.  state_rows [nrows, N] float64 is updated IN PLACE;
    x/delta/z_rows [nrows]; B, C [batch, N].  Returns y [nrows] float64."""
    dt = _DT[dtype]
    rows = np.asarray(rows, dtype=np.int64)
    nrows = len(rows)
    A = _c(A, np.float32)
    N = A.shape[1]
    if not (isinstance(state_rows, np.ndarray) and state_rows.dtype == np.float64
            and state_rows.flags.c_contiguous and state_rows.shape == (nrows, N)):
        raise TypeError("state_rows must be a C-contiguous float64 array [nrows, N]")
    rb = np.ascontiguousarray(rows // dim, dtype=np.int32)
    rd = np.ascontiguousarray(rows % dim, dtype=np.int32)
    x_rows, delta_rows, z_rows = (_storage(x, dt) for x in (x_rows, delta_rows, z_rows))
    B, C = _storage(B, dt), _storage(C, dt)
    D, delta_bias = _c(D, np.float32), _c(delta_bias, np.float32)
    y = np.empty(nrows, dtype=np.float64)
    if disc == "simple":
        rc = lib().oracle_state_step_rows(nrows, _ptr(rb), _ptr(rd), dim, N, dt, _ptr(state_rows),
                                          _ptr(x_rows), _ptr(delta_rows), _ptr(z_rows), _ptr(A),
                                          _ptr(D), _ptr(delta_bias), _ptr(B), _ptr(C),
                                          int(bool(softplus)), _ptr(y), int(nthreads))
    else:
        rc = lib().oracle_state_step_rows_ex(nrows, _ptr(rb), _ptr(rd), dim, N, dt,
                                             _ptr(state_rows), _ptr(x_rows), _ptr(delta_rows),
                                             _ptr(z_rows), _ptr(A), _ptr(D), _ptr(delta_bias),
                                             _ptr(B), _ptr(C), int(bool(softplus)), DISC[disc],
                                             _ptr(y), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_state_step_rows rejected its arguments (rc={rc})")
    return y


def state_step(state, x, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True,
               dtype="f32", nthreads=0, disc="simple"):
    """Full decode step.  state [batch, dim, N] float64 updated in place; x/delta/z [batch, dim];
    B, C [batch, N].  Returns y [batch, dim] float64."""
    bsz, dim, N = state.shape
    rows = np.arange(bsz * dim)
    st = state.reshape(bsz * dim, N)
    r = lambda a: None if a is None else np.asarray(a).reshape(bsz * dim)
    y = state_step_rows(rows, dim, st, r(x), r(delta), r(z), A, D, delta_bias, B, C, softplus,
                        dtype, nthreads, disc)
    return y.reshape(bsz, dim)


def scan_bwd_rows(rows, batch, dim, u_rows, delta_rows, z_rows, A, D, delta_bias, B, C, dy_rows,
                  softplus=True, dtype="f32", h0_rows=None, dstate_rows=None, disc="simple",
                  nthreads=0):
    """Gradients of the scan for the channels ``rows``: the loss is sum(dy * y) +
    sum(dstate * last_state) over those channels.  Returns a dict of float64 arrays: per channel
    du, ddelta, dz (None without z), dh0 [nrows, N]; summed over the given channels dA [dim, N],
    dD [dim], ddelta_bias [dim], dB, dC [batch, N, L]."""
    dt = _DT[dtype]
    rows = np.asarray(rows, dtype=np.int64)
    nrows = len(rows)
    A = _c(A, np.float32)
    N = A.shape[1]
    L = np.asarray(u_rows).shape[-1]
    rb = np.ascontiguousarray(rows // dim, dtype=np.int32)
    rd = np.ascontiguousarray(rows % dim, dtype=np.int32)
    has_z = z_rows is not None
    u_rows, delta_rows, z_rows = (_storage(x, dt) for x in (u_rows, delta_rows, z_rows))
    B, C = _storage(B, dt), _storage(C, dt)
    D, delta_bias = _c(D, np.float32), _c(delta_bias, np.float32)
    h0, dyr, dst = _c(h0_rows, np.float64), _c(dy_rows, np.float64), _c(dstate_rows, np.float64)
    out = {"du": np.empty((nrows, L)), "ddelta": np.empty((nrows, L)),
           "dz": np.empty((nrows, L)) if has_z else None, "dh0": np.empty((nrows, N)),
           "dA": np.zeros((A.shape[0], N)), "dD": np.zeros(A.shape[0]),
           "ddelta_bias": np.zeros(A.shape[0]), "dB": np.zeros((batch, N, L)),
           "dC": np.zeros((batch, N, L))}
    rc = lib().oracle_scan_bwd_rows(
        nrows, _ptr(rb), _ptr(rd), batch, dim, N, L, dt, _ptr(u_rows), _ptr(delta_rows),
        _ptr(z_rows), _ptr(A), _ptr(D), _ptr(delta_bias), _ptr(B), _ptr(C), int(bool(softplus)),
        DISC[disc], _ptr(h0), _ptr(dyr), _ptr(dst), _ptr(out["du"]), _ptr(out["ddelta"]),
        _ptr(out["dz"]), _ptr(out["dh0"]), _ptr(out["dA"]), _ptr(out["dD"]),
        _ptr(out["ddelta_bias"]), _ptr(out["dB"]), _ptr(out["dC"]), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_scan_bwd_rows rejected its arguments (rc={rc})")
    return out


def scan_bwd(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, softplus=True, dtype="f32",
             h0=None, dlast_state=None, disc="simple", nthreads=0):
    """Gradients of the full scan.  u, delta, z, dy [batch, dim, L]; dlast_state [batch, dim, N]
    (None = 0).  Returns a dict: du, ddelta, dz [batch, dim, L], dh0 [batch, dim, N], dA [dim, N],
    dD, ddelta_bias [dim], dB, dC [batch, N, L] (float64)."""
    bsz, dim, L = np.asarray(u).shape
    N = np.asarray(A).shape[1]
    r = lambda x, w: None if x is None else np.asarray(x).reshape(bsz * dim, w)
    out = scan_bwd_rows(np.arange(bsz * dim), bsz, dim, r(u, L), r(delta, L), r(z, L), A, D,
                        delta_bias, B, C, r(np.asarray(dy, np.float64), L), softplus, dtype,
                        r(h0, N), r(dlast_state, N), disc, nthreads)
    for k in ("du", "ddelta", "dz"):
        if out[k] is not None:
            out[k] = out[k].reshape(bsz, dim, L)
    out["dh0"] = out["dh0"].reshape(bsz, dim, N)
    return out


def causal_conv_rows(rows, dim, x_rows, w, conv_bias=None, silu=True, dtype="f32", x_prev_rows=None):
    """Causal depthwise convolution of the channels ``rows`` (flat b*dim + d): x_rows [nrows, L]
    in storage dtype, w [dim, K], conv_bias [dim]; x_prev_rows [nrows, K-1] (the inputs before
    position 0, oldest first; None = zeros).  Returns u [nrows, L] float64."""
    dt = _DT[dtype]
    rows = np.asarray(rows, dtype=np.int64)
    w = _c(w, np.float32)
    K = w.shape[1]
    L = np.asarray(x_rows).shape[-1]
    rd = np.ascontiguousarray(rows % dim, dtype=np.int32)
    x_rows = _storage(x_rows, dt)
    prev = _c(x_prev_rows, np.float64)
    u = np.empty((len(rows), L), dtype=np.float64)
    rc = lib().oracle_causal_conv_rows(len(rows), _ptr(rd), dim, K, L, dt, _ptr(x_rows), _ptr(w),
                                       _ptr(_c(conv_bias, np.float32)), int(bool(silu)), _ptr(prev), _ptr(u))
    if rc != 0:
        raise ValueError(f"oracle_causal_conv_rows rejected its arguments (rc={rc})")
    return u


def causal_conv(x, w, conv_bias=None, silu=True, dtype="f32", x_prev=None):
    """Full causal depthwise convolution: x [batch, dim, L] -> u [batch, dim, L] float64;
    x_prev [batch, dim, K-1] or None."""
    bsz, dim, L = np.asarray(x).shape
    K = np.asarray(w).shape[1]
    prev = None if x_prev is None else np.asarray(x_prev, np.float64).reshape(bsz * dim, K - 1)
    u = causal_conv_rows(np.arange(bsz * dim), dim, np.asarray(x).reshape(bsz * dim, L), w, conv_bias, silu,
                         dtype, prev)
    return u.reshape(bsz, dim, L)


def _as_f64(x, dtype):
    """Storage values as float64: bf16 bit patterns widened exactly, fp32 / float64 as they are."""
    if dtype == "bf16":
        bits = np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16
        return bits.view(np.float32).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def causal_conv_bwd(x, w, du, conv_bias=None, silu=True, dtype="f32", x_prev=None):
    """Gradients of the causal depthwise convolution ``causal_conv`` computes, for the loss
    sum(du * u).  x [batch, dim, L] in storage dtype ("f32", "bf16", or "f64" for float64 values);
    w [dim, K]; du [batch, dim, L] (float64); conv_bias [dim] or None; x_prev [batch, dim, K-1] (the
    inputs before position 0, oldest first) or None (zeros).

    The convolution in front of the SSM (visual guide, section 3.5) is
        pre[t] = conv_bias + sum_{k<K} w[k] x[t-(K-1)+k],   u[t] = silu(pre[t]) (or pre[t]),
    so by the chain rule, with s the logistic function and silu'(p) = s(p) (1 + p (1 - s(p))):
        dpre[t] = du[t] silu'(pre[t])                   (du[t] without the activation)
        dx[j]   = sum_k w[k] dpre[j + (K-1) - k]        (terms with the index inside [0, L))
        dw[k]   = sum over batch and t of dpre[t] x[t-(K-1)+k]
        dbias   = sum over batch and t of dpre[t]
    and dx_prev the dx formula at the K-1 positions before 0.  Returns float64 arrays dx
    [batch, dim, L], dw [dim, K], dconv_bias [dim], dx_prev [batch, dim, K-1]."""
    xs = _as_f64(x, dtype)
    bsz, dim, L = xs.shape
    w = np.asarray(w, dtype=np.float64)
    K = w.shape[1]
    du = np.asarray(du, dtype=np.float64)
    bias = np.zeros(dim) if conv_bias is None else np.asarray(conv_bias, dtype=np.float64)
    prev = np.zeros((bsz, dim, K - 1)) if x_prev is None else np.asarray(x_prev, dtype=np.float64)
    # xe[..., i] = x at position i - (K-1): the K-1 inputs before the sequence, then the sequence
    xe = np.concatenate([prev, xs], axis=2)
    pre = np.broadcast_to(bias[None, :, None], (bsz, dim, L)).copy()
    for k in range(K):
        pre += w[None, :, k, None] * xe[:, :, k:k + L]
    if silu:
        s = 1.0 / (1.0 + np.exp(-pre))
        dpre = du * s * (1.0 + pre * (1.0 - s))
    else:
        dpre = du.copy()
    dxe = np.zeros((bsz, dim, L + K - 1))
    dw = np.zeros((dim, K))
    for k in range(K):
        dxe[:, :, k:k + L] += w[None, :, k, None] * dpre
        dw[:, k] = np.sum(dpre * xe[:, :, k:k + L], axis=(0, 2))
    return {"dx": dxe[:, :, K - 1:], "dw": dw, "dconv_bias": np.sum(dpre, axis=(0, 2)),
            "dx_prev": dxe[:, :, :K - 1]}
