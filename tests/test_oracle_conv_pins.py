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
