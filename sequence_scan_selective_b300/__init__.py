"""B300-native selective scan (the core of Mamba's selective SSM layer) behind libmambascan.so.

This module only marshals arguments: it checks torch tensors (device memory), passes their data
pointers and the current CUDA stream to the library, and raises on a negative status.  Every step of
the computation runs in the library's sm_103a kernels; there is no fallback.  If the compiled
library is missing, importing this package raises ImportError.

Entry points (names as in include/mamba_scan.h):
  mamba_scan_fwd(u, delta, A, B, C, D, z, delta_bias, softplus, y=None, last_state=None, h0=None,
                 disc="simple")   (h0 -> mamba_scan_fwd_state; disc="zoh" -> mamba_scan_fwd_ex)
  mamba_scan_fwd_noalloc(...)   same arguments; the library allocates no device memory
  mamba_scan_fwd_pipelined(...)  the scan of host-resident inputs, batch rows pipelined over streams
  mamba_state_step(state, x, delta, A, B, C, D, z, delta_bias, softplus, y=None)
  mamba_scan_bwd(u, delta, A, B, C, dy, D, z, delta_bias, softplus, h0=None, dlast_state=None,
                 ckpt=None)     (ckpt -> mamba_scan_bwd_ckpt)
  mamba_scan_fwd_train(...)     mamba_scan_fwd that also returns the backward pass's checkpoints
  train_checkpoint_bytes(u, A)  their size (mamba_scan_fwd_train_ckpt_bytes; 0: none kept)
  mamba_scan_fwd_conv(...), mamba_scan_bwd_conv(...)   with the block's causal convolution
  selective_scan(u, delta, A, B, C, D, z, delta_bias, softplus, h0=None, disc="simple",
                 checkpoints=True)   the scan as an autograd operation (forward + backward above)
  selective_scan_conv(...)      the same with the convolution in front
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmambascan.so")

MAMBA_F32, MAMBA_BF16 = 0, 1
MAMBA_OK, MAMBA_ERR_ARG, MAMBA_ERR_CUDA, MAMBA_ERR_TIMEOUT = 0, -1, -2, -3
MAX_DSTATE = 64


class MambaScanError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("dim", ctypes.c_int), ("dstate", ctypes.c_int),
                ("seqlen", ctypes.c_longlong), ("in_dtype", ctypes.c_int)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmambascan.so is not built ({LIB_PATH}); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'` or "
                          "`python sequence_scan_selective_b300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I = ctypes.c_void_p, ctypes.c_int
    for name in ("mamba_scan_fwd", "mamba_scan_fwd_noalloc"):
        getattr(lib, name).restype = I
        getattr(lib, name).argtypes = [ctypes.POINTER(Shape), P, P, P, P, P, P, P, P, I, P, P, P]
    lib.mamba_scan_fwd_state.restype = I
    lib.mamba_scan_fwd_state.argtypes = [ctypes.POINTER(Shape), P, P, P, P, P, P, P, P, I, P, P, P, P]
    lib.mamba_scan_fwd_ex.restype = I
    lib.mamba_scan_fwd_ex.argtypes = [ctypes.POINTER(Shape), I, P, P, P, P, P, P, P, P, I, P, P, P, P]
    lib.mamba_scan_fwd_conv.restype = I
    lib.mamba_scan_fwd_conv.argtypes = [ctypes.POINTER(Shape), I, P, P, P, I, I, P, P, P, P, P, P, P, P, I, P, P, P,
                                        P]
    lib.mamba_state_step_ex.restype = I
    lib.mamba_state_step_ex.argtypes = [ctypes.POINTER(Shape), I, P, P, P, P, P, P, P, P, P, I, P, P]
    lib.mamba_state_step.restype = I
    lib.mamba_state_step.argtypes = [ctypes.POINTER(Shape), P, P, P, P, P, P, P, P, P, I, P, P]
    lib.mamba_scan_bwd.restype = I
    lib.mamba_scan_bwd.argtypes = [ctypes.POINTER(Shape), I] + [P] * 8 + [I] + [P] * 13
    lib.mamba_scan_fwd_train.restype = I
    lib.mamba_scan_fwd_train.argtypes = [ctypes.POINTER(Shape), I] + [P] * 8 + [I] + [P] * 6
    lib.mamba_scan_fwd_train_ckpt_bytes.restype = I
    lib.mamba_scan_fwd_train_ckpt_bytes.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(ctypes.c_size_t)]
    lib.mamba_scan_bwd_ckpt.restype = I
    lib.mamba_scan_bwd_ckpt.argtypes = [ctypes.POINTER(Shape), I] + [P] * 8 + [I] + [P] * 14
    lib.mamba_scan_bwd_conv.restype = I
    lib.mamba_scan_bwd_conv.argtypes = [ctypes.POINTER(Shape), I, P, P, P, I, I, P] + [P] * 7 + [I] + [P] * 16
    lib.mamba_scan_last_error.restype = ctypes.c_char_p
    lib.mamba_scan_last_error.argtypes = []
    lib.mamba_scan_version.restype = I
    lib.mamba_scan_version.argtypes = []
    lib.mamba_scan_device_status.restype = I
    lib.mamba_scan_device_status.argtypes = [P]
    lib.mamba_scan_launch_count.restype = ctypes.c_longlong
    lib.mamba_scan_launch_count.argtypes = []
    return lib


_lib = _load()

# symbols the header declares; the tests check that every one of them is exported
EXPORTED = ("mamba_scan_fwd", "mamba_scan_fwd_noalloc", "mamba_scan_fwd_state", "mamba_scan_fwd_ex",
            "mamba_scan_fwd_conv", "mamba_state_step", "mamba_state_step_ex", "mamba_scan_bwd", "mamba_scan_bwd_conv",
            "mamba_scan_fwd_train", "mamba_scan_bwd_ckpt", "mamba_scan_fwd_train_ckpt_bytes",
            "mamba_scan_last_error", "mamba_scan_version", "mamba_scan_device_status",
            "mamba_scan_launch_count")
MAMBA_DISC_SIMPLE, MAMBA_DISC_ZOH = 0, 1
_DISC = {"simple": MAMBA_DISC_SIMPLE, "zoh": MAMBA_DISC_ZOH}


def lib() -> ctypes.CDLL:
    return _lib


def _check(rc: int) -> None:
    if rc != MAMBA_OK:
        raise MambaScanError(rc, _lib.mamba_scan_last_error().decode(errors="replace"))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MAMBA_F32
    if t.dtype == torch.bfloat16:
        return MAMBA_BF16
    raise TypeError(f"unsupported storage dtype {t.dtype}; use float32 or bfloat16")


def _ptr(t: Optional[torch.Tensor], shape, dtype, name: str):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device=None) -> ctypes.c_void_p:
    if stream is None:
        if _raw_stream is not None:
            idx = device.index if device is not None and device.index is not None else torch.cuda.current_device()
            return ctypes.c_void_p(_raw_stream(idx))
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class PreparedCall:
    """A validated call into the library: the argument tuple is built once, so each launch costs
    only the C call (tensor checks, shape struct and stream lookup are not repeated).  The tensors
    passed at preparation must stay alive and in place while the object is used."""

    def __init__(self, fn, args, keep):
        self._fn, self._args, self._keep = fn, args, keep

    def __call__(self) -> None:
        rc = self._fn(*self._args)
        if rc != MAMBA_OK:
            _check(rc)


def mamba_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, y=None,
                   last_state=None, want_state=True, stream=None, h0=None, disc="simple"):
    """Selective scan.  u, delta, z [b, d, L]; B, C [b, N, L] (float32 or bfloat16, all the same);
    A [d, N], D [d], delta_bias [d] float32; h0 [b, d, N] float32 initial state (None = zero; it may
    be the last_state tensor itself); disc "simple" (Bbar = Delta B) or "zoh" (exact zero-order
    hold).  Returns (y [b, d, L] in the input dtype, last_state [b, d, N] float32 or None)."""
    if disc != "simple":
        return _scan(_lib.mamba_scan_fwd_ex, u, delta, A, B, C, D, z, delta_bias, softplus, y, last_state,
                     want_state, stream, h0, disc)
    if h0 is not None:
        return _scan(_lib.mamba_scan_fwd_state, u, delta, A, B, C, D, z, delta_bias, softplus, y, last_state,
                     want_state, stream, h0)
    return _scan(_lib.mamba_scan_fwd, u, delta, A, B, C, D, z, delta_bias, softplus, y, last_state,
                 want_state, stream)


def mamba_scan_fwd_conv(x, conv_w, conv_bias, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True,
                        conv_silu=True, conv_prev=None, h0=None, disc="simple", y=None, last_state=None,
                        want_state=True, stream=None):
    """The scan with the block's causal depthwise convolution fused in front: x [b, d, L] (input
    dtype) replaces u, conv_w [d, K] (K <= 4) and conv_bias [d] float32, conv_prev [b, d, K-1]
    float32 (inputs before position 0, or None).  Other arguments and the result as for
    mamba_scan_fwd."""
    args, _shape, y, last_state = _conv_args(x, conv_w, conv_bias, delta, A, B, C, D, z, delta_bias, softplus,
                                             conv_silu, conv_prev, h0, disc, y, last_state, want_state, stream)
    _check(_lib.mamba_scan_fwd_conv(*args))
    return y, last_state


def prepare_scan_fwd_conv(x, conv_w, conv_bias, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True,
                          conv_silu=True, conv_prev=None, h0=None, disc="simple", y=None, last_state=None,
                          want_state=True, stream=None):
    """mamba_scan_fwd_conv with its arguments checked once.  Returns (call, y, last_state)."""
    args, shape, y, last_state = _conv_args(x, conv_w, conv_bias, delta, A, B, C, D, z, delta_bias, softplus,
                                            conv_silu, conv_prev, h0, disc, y, last_state, want_state, stream)
    keep = (shape, x, conv_w, conv_bias, conv_prev, delta, A, B, C, D, z, delta_bias, h0, y, last_state)
    return PreparedCall(_lib.mamba_scan_fwd_conv, args, keep), y, last_state


def _conv_args(x, conv_w, conv_bias, delta, A, B, C, D, z, delta_bias, softplus, conv_silu, conv_prev, h0, disc,
               y, last_state, want_state, stream):
    bsz, dim, L = x.shape
    N = A.shape[1]
    K = conv_w.shape[1]
    dt = x.dtype
    if y is None:
        y = torch.empty_like(x)
    if last_state is None and want_state:
        last_state = torch.empty((bsz, dim, N), device=x.device, dtype=torch.float32)
    shape = Shape(bsz, dim, N, L, _dtype_code(x))
    args = (ctypes.byref(shape), _DISC[disc], _ptr(x, (bsz, dim, L), dt, "x"),
            _ptr(conv_w, (dim, K), torch.float32, "conv_w"), _ptr(conv_bias, (dim,), torch.float32, "conv_bias"),
            int(K), int(bool(conv_silu)), _ptr(conv_prev, (bsz, dim, K - 1), torch.float32, "conv_prev"),
            _ptr(delta, (bsz, dim, L), dt, "delta"), _ptr(A, (dim, N), torch.float32, "A"),
            _ptr(B, (bsz, N, L), dt, "B"), _ptr(C, (bsz, N, L), dt, "C"), _ptr(D, (dim,), torch.float32, "D"),
            _ptr(z, (bsz, dim, L), dt, "z"), _ptr(delta_bias, (dim,), torch.float32, "delta_bias"),
            int(bool(softplus)), _ptr(h0, (bsz, dim, N), torch.float32, "h0"), _ptr(y, (bsz, dim, L), dt, "y"),
            _ptr(last_state, (bsz, dim, N), torch.float32, "last_state"), _stream(stream, x.device))
    return args, shape, y, last_state


def mamba_scan_fwd_noalloc(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, y=None,
                           last_state=None, want_state=True, stream=None):
    """The same scan through the allocation-free entry point: the library itself allocates no
    device memory (split-sequence carries use its fixed scratch array).  Pass y and last_state to
    keep this wrapper from allocating them with torch."""
    return _scan(_lib.mamba_scan_fwd_noalloc, u, delta, A, B, C, D, z, delta_bias, softplus, y, last_state,
                 want_state, stream)


def _scan_args(fn, u, delta, A, B, C, D, z, delta_bias, softplus, y, last_state, want_state, stream, h0=None,
               disc="simple"):
    bsz, dim, L = u.shape
    N = A.shape[1]
    dt = u.dtype
    code = _dtype_code(u)
    if y is None:
        y = torch.empty_like(u)
    if last_state is None and want_state:
        last_state = torch.empty((bsz, dim, N), device=u.device, dtype=torch.float32)
    shape = Shape(bsz, dim, N, L, code)
    lead = (ctypes.byref(shape), _DISC[disc]) if fn is _lib.mamba_scan_fwd_ex else (ctypes.byref(shape),)
    args = lead + (
        _ptr(u, (bsz, dim, L), dt, "u"), _ptr(delta, (bsz, dim, L), dt, "delta"),
        _ptr(A, (dim, N), torch.float32, "A"), _ptr(B, (bsz, N, L), dt, "B"),
        _ptr(C, (bsz, N, L), dt, "C"), _ptr(D, (dim,), torch.float32, "D"),
        _ptr(z, (bsz, dim, L), dt, "z"), _ptr(delta_bias, (dim,), torch.float32, "delta_bias"),
        int(bool(softplus)))
    if fn is _lib.mamba_scan_fwd_state or fn is _lib.mamba_scan_fwd_ex:
        args = args + (_ptr(h0, (bsz, dim, N), torch.float32, "h0"),)
    args = args + (_ptr(y, (bsz, dim, L), dt, "y"), _ptr(last_state, (bsz, dim, N), torch.float32, "last_state"),
                   _stream(stream, u.device))
    return args, shape, y, last_state


def _scan(fn, u, delta, A, B, C, D, z, delta_bias, softplus, y, last_state, want_state, stream, h0=None,
          disc="simple"):
    args, _shape, y, last_state = _scan_args(fn, u, delta, A, B, C, D, z, delta_bias, softplus, y, last_state,
                                             want_state, stream, h0, disc)
    _check(fn(*args))
    return y, last_state


def train_checkpoint_bytes(u, A) -> int:
    """Bytes of the checkpoints mamba_scan_fwd_train keeps for u [b, d, L] and A [d, N] on the
    current device: 8 per (batch row, channel, step), or 0 when it keeps none."""
    bsz, dim, L = u.shape
    nbytes = ctypes.c_size_t(0)
    with (torch.cuda.device(u.device) if u.is_cuda else contextlib.nullcontext()):
        _check(_lib.mamba_scan_fwd_train_ckpt_bytes(ctypes.byref(Shape(bsz, dim, A.shape[1], L, _dtype_code(u))),
                                                    ctypes.byref(nbytes)))
    return nbytes.value


def mamba_scan_fwd_train(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, h0=None, disc="simple",
                         y=None, last_state=None, ckpt=None, stream=None):
    """Forward pass of training (d_state <= 16): mamba_scan_fwd that also writes the state before
    every 8-position slot, ckpt [b, ceil(L/8), d, 16] float32, for mamba_scan_bwd(..., ckpt=...).
    Returns (y, last_state, ckpt), with ckpt None when the library splits the sequence along L and
    keeps no checkpoints (then no buffer is allocated for them)."""
    bsz, dim, L = u.shape
    if ckpt is None:
        if train_checkpoint_bytes(u, A) == 0:
            y, last_state = _scan(_lib.mamba_scan_fwd_ex, u, delta, A, B, C, D, z, delta_bias, softplus, y,
                                  last_state, True, stream, h0, disc)
            return y, last_state, None
        ckpt = torch.empty((bsz, (L + 7) // 8, dim, 16), device=u.device, dtype=torch.float32)
    args, _shape, y, last_state = _scan_args(_lib.mamba_scan_fwd_ex, u, delta, A, B, C, D, z, delta_bias, softplus,
                                             y, last_state, True, stream, h0, disc)
    written = ctypes.c_int(0)
    args = args[:-1] + (_ptr(ckpt, (bsz, (L + 7) // 8, dim, 16), torch.float32, "ckpt"), ctypes.byref(written),
                        args[-1])
    _check(_lib.mamba_scan_fwd_train(*args))
    return y, last_state, (ckpt if written.value else None)


def prepare_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, y=None,
                     last_state=None, want_state=True, stream=None, noalloc=False, disc="simple"):
    """mamba_scan_fwd (or mamba_scan_fwd_noalloc; mamba_scan_fwd_ex for disc="zoh") with its
    arguments checked once.  Returns (call, y, last_state); call() enqueues the scan on the stream
    current at preparation."""
    if disc != "simple":
        if noalloc:
            raise ValueError("the allocation-free entry point takes the simplified discretisation only")
        fn = _lib.mamba_scan_fwd_ex
    else:
        fn = _lib.mamba_scan_fwd_noalloc if noalloc else _lib.mamba_scan_fwd
    args, shape, y, last_state = _scan_args(fn, u, delta, A, B, C, D, z, delta_bias, softplus, y, last_state,
                                            want_state, stream, None, disc)
    keep = (shape, u, delta, A, B, C, D, z, delta_bias, y, last_state)
    return PreparedCall(fn, args, keep), y, last_state


def _step_args(state, x, delta, A, B, C, D, z, delta_bias, softplus, y, stream, disc="simple"):
    bsz, dim, N = state.shape
    dt = x.dtype
    code = _dtype_code(x)
    if y is None:
        y = torch.empty_like(x)
    shape = Shape(bsz, dim, N, 1, code)
    lead = (ctypes.byref(shape),) if disc == "simple" else (ctypes.byref(shape), _DISC[disc])
    args = lead + (
        _ptr(state, (bsz, dim, N), torch.float32, "state"),
        _ptr(x, (bsz, dim), dt, "x"), _ptr(delta, (bsz, dim), dt, "delta"),
        _ptr(A, (dim, N), torch.float32, "A"), _ptr(B, (bsz, N), dt, "B"), _ptr(C, (bsz, N), dt, "C"),
        _ptr(D, (dim,), torch.float32, "D"), _ptr(z, (bsz, dim), dt, "z"),
        _ptr(delta_bias, (dim,), torch.float32, "delta_bias"), int(bool(softplus)),
        _ptr(y, (bsz, dim), dt, "y"), _stream(stream, state.device))
    return args, shape, y


def mamba_state_step(state, x, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, y=None,
                     stream=None, disc="simple"):
    """One decode step.  state [b, d, N] float32 (updated in place); x, delta, z [b, d];
    B, C [b, N]; disc as for mamba_scan_fwd; returns y [b, d] in the input dtype."""
    args, _shape, y = _step_args(state, x, delta, A, B, C, D, z, delta_bias, softplus, y, stream, disc)
    _check((_lib.mamba_state_step if disc == "simple" else _lib.mamba_state_step_ex)(*args))
    return y


def prepare_state_step(state, x, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, y=None,
                       stream=None, disc="simple"):
    """mamba_state_step (mamba_state_step_ex for disc="zoh") with its arguments checked once.
    Returns (call, y)."""
    args, shape, y = _step_args(state, x, delta, A, B, C, D, z, delta_bias, softplus, y, stream, disc)
    keep = (shape, state, x, delta, A, B, C, D, z, delta_bias, y)
    fn = _lib.mamba_state_step if disc == "simple" else _lib.mamba_state_step_ex
    return PreparedCall(fn, args, keep), y


def _bwd_args(u, delta, A, B, C, dy, D, z, delta_bias, softplus, h0, dlast_state, disc, stream, out):
    bsz, dim, L = u.shape
    N = A.shape[1]
    dt = u.dtype
    code = _dtype_code(u)
    f32 = dict(device=u.device, dtype=torch.float32)
    if out is None:
        out = {"du": torch.empty_like(u), "ddelta": torch.empty_like(u),
               "dz": torch.empty_like(u) if z is not None else None,
               "dA": torch.empty((dim, N), **f32), "dB": torch.empty((bsz, N, L), **f32),
               "dC": torch.empty((bsz, N, L), **f32),
               "dD": torch.empty((dim,), **f32) if D is not None else None,
               "ddelta_bias": torch.empty((dim,), **f32) if delta_bias is not None else None,
               "dh0": torch.empty((bsz, dim, N), **f32) if h0 is not None else None}
    shape = Shape(bsz, dim, N, L, code)
    args = (
        ctypes.byref(shape), _DISC[disc], _ptr(u, (bsz, dim, L), dt, "u"),
        _ptr(delta, (bsz, dim, L), dt, "delta"), _ptr(A, (dim, N), torch.float32, "A"),
        _ptr(B, (bsz, N, L), dt, "B"), _ptr(C, (bsz, N, L), dt, "C"),
        _ptr(D, (dim,), torch.float32, "D"), _ptr(z, (bsz, dim, L), dt, "z"),
        _ptr(delta_bias, (dim,), torch.float32, "delta_bias"), int(bool(softplus)),
        _ptr(h0, (bsz, dim, N), torch.float32, "h0"), _ptr(dy, (bsz, dim, L), dt, "dy"),
        _ptr(dlast_state, (bsz, dim, N), torch.float32, "dlast_state"),
        _ptr(out["du"], (bsz, dim, L), dt, "du"), _ptr(out["ddelta"], (bsz, dim, L), dt, "ddelta"),
        _ptr(out["dz"], (bsz, dim, L), dt, "dz"), _ptr(out["dA"], (dim, N), torch.float32, "dA"),
        _ptr(out["dB"], (bsz, N, L), torch.float32, "dB"), _ptr(out["dC"], (bsz, N, L), torch.float32, "dC"),
        _ptr(out["dD"], (dim,), torch.float32, "dD"),
        _ptr(out["ddelta_bias"], (dim,), torch.float32, "ddelta_bias"),
        _ptr(out["dh0"], (bsz, dim, N), torch.float32, "dh0"), _stream(stream, u.device))
    return args, shape, out


def mamba_scan_bwd(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, softplus=True, h0=None,
                   dlast_state=None, disc="simple", stream=None, out=None, ckpt=None):
    """Gradients of mamba_scan_fwd for the loss sum(dy * y) + sum(dlast_state * last_state).
    Inputs as for mamba_scan_fwd plus dy [b, d, L] (input dtype) and dlast_state [b, d, N] float32;
    ckpt: the checkpoints of mamba_scan_fwd_train on the same inputs, or None.
    Returns a dict: du, ddelta, dz [b, d, L] (input dtype; dz None without z), dA [d, N],
    dB, dC [b, N, L], dD, ddelta_bias [d] (None when D / delta_bias is None), dh0 [b, d, N]
    (None without h0), all float32 except du, ddelta, dz.  ``out`` may supply that dict."""
    args, _shape, out = _bwd_args(u, delta, A, B, C, dy, D, z, delta_bias, softplus, h0, dlast_state, disc,
                                  stream, out)
    if ckpt is None:
        _check(_lib.mamba_scan_bwd(*args))
    else:
        bsz, dim, L = u.shape
        # mamba_scan_bwd_ckpt takes ckpt right after dlast_state (argument 14)
        args = args[:14] + (_ptr(ckpt, (bsz, (L + 7) // 8, dim, 16), torch.float32, "ckpt"),) + args[14:]
        _check(_lib.mamba_scan_bwd_ckpt(*args))
    return out


def prepare_scan_bwd(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, softplus=True, h0=None,
                     dlast_state=None, disc="simple", stream=None, out=None, ckpt=None):
    """mamba_scan_bwd (mamba_scan_bwd_ckpt with ckpt) with its arguments checked once.  Returns
    (call, out)."""
    args, shape, out = _bwd_args(u, delta, A, B, C, dy, D, z, delta_bias, softplus, h0, dlast_state, disc,
                                 stream, out)
    keep = (shape, u, delta, A, B, C, dy, D, z, delta_bias, h0, dlast_state, out, ckpt)
    if ckpt is None:
        return PreparedCall(_lib.mamba_scan_bwd, args, keep), out
    bsz, dim, L = u.shape
    args = args[:14] + (_ptr(ckpt, (bsz, (L + 7) // 8, dim, 16), torch.float32, "ckpt"),) + args[14:]
    return PreparedCall(_lib.mamba_scan_bwd_ckpt, args, keep), out


def mamba_scan_bwd_conv(x, conv_w, conv_bias, delta, A, B, C, dy, D=None, z=None, delta_bias=None, softplus=True,
                        conv_silu=True, conv_prev=None, h0=None, dlast_state=None, disc="simple", stream=None):
    """Gradients of mamba_scan_fwd_conv (the scan with the block's causal convolution in front) for
    the loss sum(dy * y) + sum(dlast_state * last_state).  Inputs as for mamba_scan_fwd_conv plus dy
    and dlast_state as for mamba_scan_bwd.  Returns the dict of mamba_scan_bwd with du replaced by
    dx (input dtype) and three more float32 entries: dconv_w [d, K], dconv_bias [d] and dconv_prev
    [b, d, K-1] (None when K == 1)."""
    bsz, dim, L = x.shape
    N = A.shape[1]
    K = conv_w.shape[1]
    dt = x.dtype
    f32 = dict(device=x.device, dtype=torch.float32)
    out = {"dx": torch.empty_like(x), "ddelta": torch.empty_like(x),
           "dz": torch.empty_like(x) if z is not None else None,
           "dA": torch.empty((dim, N), **f32), "dB": torch.empty((bsz, N, L), **f32),
           "dC": torch.empty((bsz, N, L), **f32),
           "dD": torch.empty((dim,), **f32) if D is not None else None,
           "ddelta_bias": torch.empty((dim,), **f32) if delta_bias is not None else None,
           "dconv_w": torch.empty((dim, K), **f32), "dconv_bias": torch.empty((dim,), **f32),
           "dconv_prev": torch.empty((bsz, dim, K - 1), **f32) if K > 1 else None,
           "dh0": torch.empty((bsz, dim, N), **f32) if h0 is not None else None}
    shape = Shape(bsz, dim, N, L, _dtype_code(x))
    _check(_lib.mamba_scan_bwd_conv(
        ctypes.byref(shape), _DISC[disc], _ptr(x, (bsz, dim, L), dt, "x"),
        _ptr(conv_w, (dim, K), torch.float32, "conv_w"), _ptr(conv_bias, (dim,), torch.float32, "conv_bias"),
        int(K), int(bool(conv_silu)), _ptr(conv_prev, (bsz, dim, K - 1), torch.float32, "conv_prev"),
        _ptr(delta, (bsz, dim, L), dt, "delta"), _ptr(A, (dim, N), torch.float32, "A"),
        _ptr(B, (bsz, N, L), dt, "B"), _ptr(C, (bsz, N, L), dt, "C"), _ptr(D, (dim,), torch.float32, "D"),
        _ptr(z, (bsz, dim, L), dt, "z"), _ptr(delta_bias, (dim,), torch.float32, "delta_bias"),
        int(bool(softplus)), _ptr(h0, (bsz, dim, N), torch.float32, "h0"), _ptr(dy, (bsz, dim, L), dt, "dy"),
        _ptr(dlast_state, (bsz, dim, N), torch.float32, "dlast_state"),
        _ptr(out["dx"], (bsz, dim, L), dt, "dx"), _ptr(out["ddelta"], (bsz, dim, L), dt, "ddelta"),
        _ptr(out["dz"], (bsz, dim, L), dt, "dz"), _ptr(out["dA"], (dim, N), torch.float32, "dA"),
        _ptr(out["dB"], (bsz, N, L), torch.float32, "dB"), _ptr(out["dC"], (bsz, N, L), torch.float32, "dC"),
        _ptr(out["dD"], (dim,), torch.float32, "dD"), _ptr(out["ddelta_bias"], (dim,), torch.float32, "ddelta_bias"),
        _ptr(out["dconv_w"], (dim, K), torch.float32, "dconv_w"),
        _ptr(out["dconv_bias"], (dim,), torch.float32, "dconv_bias"),
        _ptr(out["dconv_prev"], (bsz, dim, K - 1), torch.float32, "dconv_prev"),
        _ptr(out["dh0"], (bsz, dim, N), torch.float32, "dh0"), _stream(stream, x.device)))
    return out


class _HostPipeline:
    """Device staging buffers and streams of mamba_scan_fwd_pipelined for one shape (kept between
    calls, so that steady use allocates nothing)."""

    def __init__(self, device, dim, N, L, dtype):
        f = dict(device=device, dtype=dtype)
        self.x = [{k: torch.empty((1, dim, L), **f) for k in ("u", "delta", "z")} for _ in range(2)]
        for slot in self.x:
            slot["B"] = torch.empty((1, N, L), **f)
            slot["C"] = torch.empty((1, N, L), **f)
            slot["y"] = torch.empty((1, dim, L), **f)
        self.streams = [torch.cuda.Stream(device) for _ in range(3)]  # copy in, scan, copy out
        self.key = (device, dim, N, L, dtype)


_pipelines = {}


def mamba_scan_fwd_pipelined(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, y=None,
                             last_state=None, stream=None):
    """The forward scan of inputs that live in host memory, with y copied back to host memory.

    u, delta, z [b, d, L] and B, C [b, N, L] are CPU tensors (pinned, for asynchronous copies); A, D,
    delta_bias are CUDA tensors as for mamba_scan_fwd.  y (CPU, pinned; allocated when None) receives
    the output and last_state (CUDA, [b, d, N] float32; allocated when None) the final state.  The
    batch rows go through in turn on three streams, so that the copy of one row's inputs to the
    device, the scan of the previous row (mamba_scan_fwd on that row) and the copy of the row
    before back to the host overlap; device staging is double-buffered and kept for the next call
    of the same shape.  The work is ordered after `stream` (default: the current stream) and the
    current stream waits for all of it, so y may be read after synchronising that stream."""
    bsz, dim, L = u.shape
    N = A.shape[1]
    dev = A.device
    cur = stream if stream is not None else torch.cuda.current_stream(dev)
    key = (dev, dim, N, L, u.dtype)
    pipe = _pipelines.get(key)
    if pipe is None:
        pipe = _pipelines[key] = _HostPipeline(dev, dim, N, L, u.dtype)
    if y is None:
        y = torch.empty_like(u).pin_memory()
    if last_state is None:
        last_state = torch.empty((bsz, dim, N), device=dev, dtype=torch.float32)
    s_in, s_scan, s_out = pipe.streams
    for s_ in pipe.streams:
        s_.wait_stream(cur)
    scanned = [None, None]   # per slot: event after the scan that last used it
    copied_out = [None, None]  # per slot: event after the copy-out that last read its y
    for i in range(bsz):
        slot = i % 2
        buf = pipe.x[slot]
        with torch.cuda.stream(s_in):
            if scanned[slot] is not None:
                s_in.wait_event(scanned[slot])
            for k, src in (("u", u), ("delta", delta), ("z", z), ("B", B), ("C", C)):
                if src is not None:
                    buf[k].copy_(src[i:i + 1], non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(s_in)
        with torch.cuda.stream(s_scan):
            s_scan.wait_event(ready)
            if copied_out[slot] is not None:
                s_scan.wait_event(copied_out[slot])
            mamba_scan_fwd(buf["u"], buf["delta"], A, buf["B"], buf["C"], D, buf["z"] if z is not None else None,
                           delta_bias, softplus, y=buf["y"], last_state=last_state[i:i + 1], stream=s_scan)
            done = torch.cuda.Event()
            done.record(s_scan)
            scanned[slot] = done
        with torch.cuda.stream(s_out):
            s_out.wait_event(done)
            y[i:i + 1].copy_(buf["y"], non_blocking=True)
            out = torch.cuda.Event()
            out.record(s_out)
            copied_out[slot] = out
    cur.wait_stream(s_scan)
    cur.wait_stream(s_out)
    return y, last_state


class _SelectiveScan(torch.autograd.Function):
    """The scan as an autograd operation: the forward pass is mamba_scan_fwd_train (d_state <= 16:
    it also keeps the state before every 8-position slot) or mamba_scan_fwd, the backward pass
    mamba_scan_bwd, which recomputes the states between those checkpoints."""

    @staticmethod
    def forward(ctx, u, delta, A, B, C, D, z, delta_bias, h0, softplus, disc, checkpoints):
        ckpt = None
        if checkpoints and A.shape[1] <= 16 and u.shape[2] > 0:  # keep what the backward pass would recompute
            y, last_state, ckpt = mamba_scan_fwd_train(u, delta, A, B, C, D, z, delta_bias, softplus, h0=h0, disc=disc)
        else:
            y, last_state = mamba_scan_fwd(u, delta, A, B, C, D, z, delta_bias, softplus, h0=h0, disc=disc)
        ctx.save_for_backward(u, delta, A, B, C, D, z, delta_bias, h0, ckpt)
        ctx.softplus, ctx.disc = softplus, disc
        return y, last_state

    @staticmethod
    def backward(ctx, dy, dlast_state):
        u, delta, A, B, C, D, z, delta_bias, h0, ckpt = ctx.saved_tensors
        dy = torch.zeros_like(u) if dy is None else dy.contiguous()
        dlast_state = None if dlast_state is None else dlast_state.contiguous()
        g = mamba_scan_bwd(u, delta, A, B, C, dy, D, z, delta_bias, ctx.softplus, h0=h0, dlast_state=dlast_state,
                           disc=ctx.disc, ckpt=ckpt)
        like = lambda t, ref: None if t is None else t.to(ref.dtype)  # dB, dC come as fp32
        return (g["du"], g["ddelta"], g["dA"], like(g["dB"], B), like(g["dC"], C), g["dD"], g["dz"],
                g["ddelta_bias"], g["dh0"], None, None, None)


def selective_scan(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, h0=None, disc="simple",
                   checkpoints=True):
    """(y, last_state) of the scan, differentiable with respect to u, delta, A, B, C, D, z,
    delta_bias and h0 (backward pass: mamba_scan_bwd).  Arguments as for mamba_scan_fwd.
    checkpoints: for d_state <= 16, the forward pass keeps the state before every 8-step slot for
    the backward pass (8 bytes per batch row, channel and step, held until the backward pass);
    False recomputes them there instead (slower step, no extra memory)."""
    return _SelectiveScan.apply(u, delta, A, B, C, D, z, delta_bias, h0, bool(softplus), disc, bool(checkpoints))


class _SelectiveScanConv(torch.autograd.Function):
    """The scan with the block's causal convolution in front, as an autograd operation: forward
    mamba_scan_fwd_conv, backward mamba_scan_bwd_conv (the convolution's output and the states are
    recomputed; only the inputs are saved)."""

    @staticmethod
    def forward(ctx, x, conv_w, conv_bias, conv_prev, delta, A, B, C, D, z, delta_bias, h0, softplus, conv_silu,
                disc):
        y, last_state = mamba_scan_fwd_conv(x, conv_w, conv_bias, delta, A, B, C, D, z, delta_bias, softplus,
                                            conv_silu=conv_silu, conv_prev=conv_prev, h0=h0, disc=disc)
        ctx.save_for_backward(x, conv_w, conv_bias, conv_prev, delta, A, B, C, D, z, delta_bias, h0)
        ctx.softplus, ctx.conv_silu, ctx.disc = softplus, conv_silu, disc
        return y, last_state

    @staticmethod
    def backward(ctx, dy, dlast_state):
        x, conv_w, conv_bias, conv_prev, delta, A, B, C, D, z, delta_bias, h0 = ctx.saved_tensors
        dy = torch.zeros_like(x) if dy is None else dy.contiguous()
        dlast_state = None if dlast_state is None else dlast_state.contiguous()
        g = mamba_scan_bwd_conv(x, conv_w, conv_bias, delta, A, B, C, dy, D, z, delta_bias, ctx.softplus,
                                conv_silu=ctx.conv_silu, conv_prev=conv_prev, h0=h0, dlast_state=dlast_state,
                                disc=ctx.disc)
        like = lambda t, ref: None if t is None or ref is None else t.to(ref.dtype)  # dB, dC come as fp32
        return (g["dx"], g["dconv_w"], like(g["dconv_bias"], conv_bias), like(g["dconv_prev"], conv_prev),
                g["ddelta"], g["dA"], like(g["dB"], B), like(g["dC"], C), g["dD"], g["dz"], g["ddelta_bias"],
                g["dh0"], None, None, None)


def selective_scan_conv(x, conv_w, conv_bias, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True,
                        conv_silu=True, conv_prev=None, h0=None, disc="simple"):
    """(y, last_state) of the scan with the block's causal convolution in front, differentiable
    with respect to x, conv_w, conv_bias, conv_prev, delta, A, B, C, D, z, delta_bias and h0
    (backward pass: mamba_scan_bwd_conv).  Arguments as for mamba_scan_fwd_conv."""
    return _SelectiveScanConv.apply(x, conv_w, conv_bias, conv_prev, delta, A, B, C, D, z, delta_bias, h0,
                                    bool(softplus), bool(conv_silu), disc)


def device_status(stream=None) -> None:
    """Synchronise and raise if a kernel abandoned a bounded wait since the last check."""
    _check(_lib.mamba_scan_device_status(_stream(stream, torch.device("cuda", torch.cuda.current_device()))))


def version() -> int:
    return _lib.mamba_scan_version()


def launch_count() -> int:
    """Kernels launched by the library in this process so far."""
    return int(_lib.mamba_scan_launch_count())
