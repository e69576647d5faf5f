"""Pins of the oracle's causal depthwise convolution (the step in front of the selective SSM in the
Mamba block: visual guide to Mamba and SSMs, section 3.5) against numpy's convolution, scipy's
logistic function, the identity kernel and the split of a sequence into two pieces."""
import numpy as np
import pytest
from scipy.special import expit

import oracle


def _case(seed, bsz=2, dim=5, L=37, K=4):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((bsz, dim, L)).astype(np.float32)
    w = rng.standard_normal((dim, K)).astype(np.float32)
    cb = rng.standard_normal(dim).astype(np.float32)
    return x, w, cb


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_conv_matches_numpy_convolve(K):
    x, w, cb = _case(1, K=K)
    u = oracle.causal_conv(x, w, cb, silu=False)
    bsz, dim, L = x.shape
    for b in range(bsz):
        for d in range(dim):
            # causal: output t sees inputs t-K+1 .. t, the newest against the last tap
            want = np.convolve(x[b, d].astype(np.float64), w[d, ::-1].astype(np.float64))[:L] + cb[d]
            np.testing.assert_allclose(u[b, d], want, rtol=1e-13, atol=1e-13)


def test_conv_activation_is_silu():
    x, w, cb = _case(2)
    lin = oracle.causal_conv(x, w, cb, silu=False)
    act = oracle.causal_conv(x, w, cb, silu=True)
    np.testing.assert_allclose(act, lin * expit(lin), rtol=1e-13, atol=1e-14)


def test_identity_kernel():
    x, _, _ = _case(3, K=1)
    u = oracle.causal_conv(x, np.ones((x.shape[1], 1), np.float32), None, silu=False)
    np.testing.assert_array_equal(u, x.astype(np.float64))


@pytest.mark.parametrize("split", [1, 3, 20])
def test_split_sequence_with_previous_inputs(split):
    x, w, cb = _case(4)
    K = w.shape[1]
    full = oracle.causal_conv(x, w, cb, silu=True)
    first = oracle.causal_conv(x[:, :, :split], w, cb, silu=True)
    prev = np.zeros(x.shape[:2] + (K - 1,), np.float64)
    tail = x[:, :, max(0, split - (K - 1)):split].astype(np.float64)
    prev[:, :, K - 1 - tail.shape[2]:] = tail
    second = oracle.causal_conv(x[:, :, split:], w, cb, silu=True, x_prev=prev)
    np.testing.assert_allclose(np.concatenate([first, second], axis=2), full, rtol=1e-14, atol=1e-15)


# ------------------------------------------------------------------------------ gradient pins
# The gradient oracle is pinned against derivatives of a forward convolution written here with
# numpy's convolve in float64 (independent of oracle.c): Richardson-extrapolated central
# differences, input by input, and for the identity activation the adjoint of the causal window,
# a full convolution of the output gradient with the same taps.

def _np_conv(x, w, cb, prev, silu):
    """u = act(cb + causal conv of [prev, x] with w), all float64, via numpy.convolve."""
    bsz, dim, L = x.shape
    K = w.shape[1]
    u = np.empty((bsz, dim, L))
    for b in range(bsz):
        for d in range(dim):
            xe = np.concatenate([prev[b, d], x[b, d]])
            pre = np.convolve(xe, w[d, ::-1])[K - 1:K - 1 + L] + cb[d]
            u[b, d] = pre * expit(pre) if silu else pre
    return u


def _richardson(f, h=1e-3):
    d1 = (f(h) - f(-h)) / (2 * h)
    d2 = (f(h / 2) - f(-h / 2)) / h
    return (4 * d2 - d1) / 3


def _grad_case(seed, K, bsz=2, dim=3, L=9):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((bsz, dim, L))
    w = rng.standard_normal((dim, K)) / np.sqrt(K)
    cb = rng.standard_normal(dim) * 0.3
    prev = rng.standard_normal((bsz, dim, K - 1))
    du = rng.standard_normal((bsz, dim, L))
    return x, w, cb, prev, du


@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("silu", [True, False])
def test_conv_gradients_match_finite_differences(K, silu):
    x, w, cb, prev, du = _grad_case(10 + K, K)
    g = oracle.causal_conv_bwd(x, w, du, cb, silu, "f64", x_prev=prev)
    loss = lambda x_, w_, cb_, p_: float(np.sum(du * _np_conv(x_, w_, cb_, p_, silu)))

    def num(arr_name, idx):
        def f(eps):
            args = {"x": x.copy(), "w": w.copy(), "cb": cb.copy(), "p": prev.copy()}
            args[arr_name][idx] += eps
            return loss(args["x"], args["w"], args["cb"], args["p"])
        return _richardson(f)

    for idx in np.ndindex(*x.shape):
        assert abs(g["dx"][idx] - num("x", idx)) <= 1e-8 * max(1.0, abs(g["dx"][idx]))
    for idx in np.ndindex(*w.shape):
        assert abs(g["dw"][idx] - num("w", idx)) <= 1e-8 * max(1.0, abs(g["dw"][idx]))
    for idx in np.ndindex(*cb.shape):
        assert abs(g["dconv_bias"][idx] - num("cb", idx)) <= 1e-8 * max(1.0, abs(g["dconv_bias"][idx]))
    for idx in np.ndindex(*prev.shape):
        assert abs(g["dx_prev"][idx] - num("p", idx)) <= 1e-8 * max(1.0, abs(g["dx_prev"][idx]))


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_conv_input_gradient_is_full_convolution(K):
    """Without the activation, input i of the extended sequence [prev, x] feeds output t through
    tap k = i - t, so its gradient is sum_k w[k] du[i - k]: numpy's full convolution of du with w."""
    x, w, cb, prev, du = _grad_case(20 + K, K, L=30)
    g = oracle.causal_conv_bwd(x, w, du, cb, False, "f64", x_prev=prev)
    bsz, dim, L = x.shape
    for b in range(bsz):
        for d in range(dim):
            got = np.concatenate([g["dx_prev"][b, d], g["dx"][b, d]])
            np.testing.assert_allclose(got, np.convolve(du[b, d], w[d]), rtol=1e-13, atol=1e-13)
