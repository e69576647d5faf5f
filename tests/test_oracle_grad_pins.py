"""Pins of the oracle's exact zero-order hold and of its gradients.

Neither check re-types the oracle's arithmetic:

* zero-order hold (visual guide to Mamba and SSMs, section 2.3: the input is held over each step of
  length Delta): the held-input ODE h' = A h + B x is integrated numerically over every step by
  scipy's DOP853 at tight tolerances and compared with the oracle's closed-form update;
* gradients (same guide, section 3.4: the backward pass recomputes the states): every gradient of
  ``oracle.scan_bwd`` is compared, input element by input element, with a Richardson-extrapolated
  central difference of the forward oracle.  The base point is dyadic (multiples of 2^-8) and the
  steps are 2^-10 and 2^-11, so every perturbed input is exact in fp32 and the difference quotient
  sees exactly the step it divides by.
"""
import numpy as np
import pytest
from scipy.integrate import solve_ivp
from scipy.special import expit

import oracle
import synth

FD_RTOL = 1e-8


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


def _dyadic(rng, shape, lo, hi):
    return (np.round(rng.uniform(lo, hi, size=shape) * 256.0) / 256.0).astype(np.float32)


def _case(seed, bsz=2, dim=3, N=3, L=7, softplus=True, gate=True, skip=True, bias=True, h0=True,
          dstate=True, zero_A=False):
    rng = np.random.default_rng(seed)
    A = _dyadic(rng, (dim, N), -2.0, -0.25)
    if zero_A:
        A[0, 1] = 0.0
    c = dict(
        u=_dyadic(rng, (bsz, dim, L), -2, 2),
        delta=_dyadic(rng, (bsz, dim, L), -2.0, 0.5) if softplus else _dyadic(rng, (bsz, dim, L), 0.05, 0.6),
        A=A, B=_dyadic(rng, (bsz, N, L), -2, 2), C=_dyadic(rng, (bsz, N, L), -2, 2),
        D=_dyadic(rng, dim, 0.5, 1.5) if skip else None,
        z=_dyadic(rng, (bsz, dim, L), -2, 2) if gate else None,
        delta_bias=_dyadic(rng, dim, -0.25, 0.25) if bias else None,
        h0=rng.normal(size=(bsz, dim, N)) if h0 else None)
    dy = rng.normal(size=(bsz, dim, L))
    ds = rng.normal(size=(bsz, dim, N)) if dstate else None
    return c, dy, ds, softplus


def _loss(c, dy, ds, softplus, disc):
    y, st = oracle.scan(c["u"], c["delta"], c["A"], c["B"], c["C"], c["D"], c["z"], c["delta_bias"],
                        softplus, "f32", h0=c["h0"], disc=disc)
    out = float(np.sum(dy * y))
    if ds is not None:
        out += float(np.sum(ds * st))
    return out


def _fd(c, dy, ds, softplus, disc, name):
    """Richardson-extrapolated central differences of the loss with respect to c[name]."""
    base = c[name]
    g = np.zeros(base.shape, np.float64)
    for idx in np.ndindex(base.shape):
        quot = []
        for eps in (2.0 ** -10, 2.0 ** -11):
            vals = []
            for sgn in (1.0, -1.0):
                p = base.copy()
                p[idx] = p[idx] + sgn * eps
                assert float(p[idx]) == float(base[idx]) + sgn * eps  # exact perturbation
                vals.append(_loss({**c, name: p}, dy, ds, softplus, disc))
            quot.append((vals[0] - vals[1]) / (2.0 * eps))
        g[idx] = (4.0 * quot[1] - quot[0]) / 3.0
    return g


CONFIGS = {
    "all_inputs": dict(),
    "bare": dict(softplus=False, gate=False, skip=False, bias=False, h0=False, dstate=False),
    "no_gate_with_state": dict(gate=False, h0=False),
    "no_softplus_gate": dict(softplus=False, skip=False),
}


@pytest.mark.parametrize("disc", ["simple", "zoh"])
@pytest.mark.parametrize("cfg", sorted(CONFIGS))
def test_gradients_match_finite_differences(cfg, disc):
    c, dy, ds, softplus = _case(11 + len(cfg), **CONFIGS[cfg])
    g = oracle.scan_bwd(c["u"], c["delta"], c["A"], c["B"], c["C"], dy, c["D"], c["z"],
                        c["delta_bias"], softplus, "f32", h0=c["h0"], dlast_state=ds, disc=disc)
    pairs = [("u", "du"), ("delta", "ddelta"), ("A", "dA"), ("B", "dB"), ("C", "dC")]
    pairs += [(k, gk) for k, gk in (("z", "dz"), ("D", "dD"), ("delta_bias", "ddelta_bias"),
                                    ("h0", "dh0")) if c[k] is not None]
    for name, gname in pairs:
        want = _fd(c, dy, ds, softplus, disc, name)
        assert _rel(g[gname], want) < FD_RTOL, (cfg, disc, gname, _rel(g[gname], want))


def test_zoh_gradients_at_zero_A():
    """A = 0 in one state: the hold factor is Delta there and its A-derivative Delta^2 / 2."""
    c, dy, ds, softplus = _case(5, zero_A=True)
    g = oracle.scan_bwd(c["u"], c["delta"], c["A"], c["B"], c["C"], dy, c["D"], c["z"],
                        c["delta_bias"], softplus, "f32", h0=c["h0"], dlast_state=ds, disc="zoh")
    for name, gname in (("A", "dA"), ("delta", "ddelta"), ("u", "du")):
        want = _fd(c, dy, ds, softplus, "zoh", name)
        assert _rel(g[gname], want) < FD_RTOL, (gname, _rel(g[gname], want))


def test_gradient_rows_sum_to_full():
    """Gradients for a subset of channels: per-channel outputs equal the full run's rows, and the
    shared gradients (dB, dC) add up over a partition of the channels."""
    c, dy, ds, softplus = _case(3, bsz=2, dim=4, N=3, L=9)
    full = oracle.scan_bwd(c["u"], c["delta"], c["A"], c["B"], c["C"], dy, c["D"], c["z"],
                           c["delta_bias"], softplus, "f32", h0=c["h0"], dlast_state=ds)
    bsz, dim, L = c["u"].shape
    N = c["A"].shape[1]
    r = lambda x, w: x.reshape(bsz * dim, w)
    parts = [np.array([0, 3, 5]), np.array([1, 2, 4, 6, 7])]
    acc_dB = np.zeros_like(full["dB"])
    for rows in parts:
        p = oracle.scan_bwd_rows(rows, bsz, dim, r(c["u"], L)[rows], r(c["delta"], L)[rows],
                                 r(c["z"], L)[rows], c["A"], c["D"], c["delta_bias"], c["B"],
                                 c["C"], r(dy, L)[rows], softplus, "f32",
                                 r(c["h0"], N)[rows], r(ds, N)[rows])
        np.testing.assert_array_equal(p["du"], r(full["du"], L)[rows])
        np.testing.assert_array_equal(p["dh0"], r(full["dh0"], N)[rows])
        acc_dB += p["dB"]
    assert _rel(acc_dB, full["dB"]) < 1e-14


def _ode_scan(c, softplus):
    """The held-input ODE h' = a h + B_t x_t, solved numerically over each step [0, Delta_t]."""
    bsz, dim, L = c["u"].shape
    N = c["A"].shape[1]
    y = np.zeros((bsz, dim, L))
    for b in range(bsz):
        for d in range(dim):
            a = c["A"][d].astype(np.float64)
            h = np.zeros(N)
            for t in range(L):
                x = float(c["u"][b, d, t])
                s = float(c["delta"][b, d, t]) + float(c["delta_bias"][d])
                dt = np.logaddexp(0.0, s) if softplus else s
                Bt = c["B"][b, :, t].astype(np.float64)
                sol = solve_ivp(lambda _t, hh: a * hh + Bt * x, (0.0, dt), h, method="DOP853",
                                rtol=1e-13, atol=1e-15)
                h = sol.y[:, -1]
                zz = float(c["z"][b, d, t])
                y[b, d, t] = (float(c["C"][b, :, t] @ h) + float(c["D"][d]) * x) * zz * expit(zz)
    return y


def test_zoh_matches_numerical_ode():
    c, _, _, softplus = _case(21, bsz=1, dim=2, N=3, L=6, h0=False)
    y, _ = oracle.scan(c["u"], c["delta"], c["A"], c["B"], c["C"], c["D"], c["z"], c["delta_bias"],
                       softplus, "f32", disc="zoh")
    assert _rel(y, _ode_scan(c, softplus)) < 1e-9


def test_zoh_and_simple_differ_at_second_order():
    """The simplified Bbar = Delta B agrees with the hold to first order in Delta: halving every
    step size quarters the gap in the first state update."""
    c, _, _, _ = _case(8, bsz=1, dim=2, N=3, L=1, softplus=False, gate=False, h0=False)
    gaps = []
    for scale in (1.0, 0.5, 0.25):
        cc = {**c, "delta": (c["delta"] * np.float32(scale)).astype(np.float32)}
        ye, _ = oracle.scan(cc["u"], cc["delta"], cc["A"], cc["B"], cc["C"], None, None, None,
                            False, "f32", disc="simple")
        yz, _ = oracle.scan(cc["u"], cc["delta"], cc["A"], cc["B"], cc["C"], None, None, None,
                            False, "f32", disc="zoh")
        gaps.append(np.max(np.abs(ye - yz)))
    assert 3.6 < gaps[0] / gaps[1] < 4.4 and 3.8 < gaps[1] / gaps[2] < 4.2, gaps


def test_zoh_equals_simple_where_A_is_zero():
    c, _, _, softplus = _case(9, zero_A=True)
    c["A"][:] = 0.0
    ye, se = oracle.scan(c["u"], c["delta"], c["A"], c["B"], c["C"], c["D"], c["z"],
                         c["delta_bias"], softplus, "f32", h0=c["h0"])
    yz, sz = oracle.scan(c["u"], c["delta"], c["A"], c["B"], c["C"], c["D"], c["z"],
                         c["delta_bias"], softplus, "f32", h0=c["h0"], disc="zoh")
    np.testing.assert_array_equal(ye, yz)
    np.testing.assert_array_equal(se, sz)


def test_zoh_decode_steps_equal_scan():
    c, _, _, softplus = _case(4, L=5)
    y, st = oracle.scan(c["u"], c["delta"], c["A"], c["B"], c["C"], c["D"], c["z"], c["delta_bias"],
                        softplus, "f32", h0=c["h0"], disc="zoh")
    state = np.array(c["h0"], np.float64, order="C")
    for t in range(c["u"].shape[2]):
        yt = oracle.state_step(state, c["u"][:, :, t], c["delta"][:, :, t], c["A"],
                               np.ascontiguousarray(c["B"][:, :, t]),
                               np.ascontiguousarray(c["C"][:, :, t]), c["D"], c["z"][:, :, t],
                               c["delta_bias"], softplus, "f32", disc="zoh")
        assert _rel(yt, y[:, :, t]) < 1e-13
    assert _rel(state, st) < 1e-13


@pytest.mark.parametrize("disc", ["simple", "zoh"])
def test_lti_input_gradient_is_a_correlation(disc):
    """Time-invariant case (constant Delta, B, C; no gate): y = K * u + D u with
    K_k = sum_n C_n Abar_n^k Bbar_n (visual guide, sections 2.5-2.7), so the gradient of
    sum_t dy_t y_t with respect to u_s is sum_{t >= s} dy_t K_{t-s} + D dy_s: a correlation of dy
    with the kernel, computed here by brute force from the closed-form kernel."""
    rng = np.random.default_rng(77)
    dim, N, L = 3, 4, 40
    A = -np.exp(rng.uniform(-1, 1, size=(dim, N))).astype(np.float32)
    dt = rng.uniform(0.05, 0.4, size=dim)
    B = rng.normal(size=(1, N, 1)).astype(np.float32).repeat(L, axis=2)
    C = rng.normal(size=(1, N, 1)).astype(np.float32).repeat(L, axis=2)
    D = rng.normal(size=dim).astype(np.float32)
    u = rng.normal(size=(1, dim, L)).astype(np.float32)
    delta = np.repeat(dt[None, :, None], L, axis=2).astype(np.float32)
    dy = rng.normal(size=(1, dim, L))
    g = oracle.scan_bwd(u, delta, A, B, C, dy, D, None, None, False, "f32", disc=disc)
    for d in range(dim):
        a = A[d].astype(np.float64)
        step = float(delta[0, d, 0])
        abar = np.exp(step * a)
        kfac = step if disc == "simple" else np.expm1(step * a) / a
        bbar = kfac * B[0, :, 0].astype(np.float64)
        K = np.array([np.sum(C[0, :, 0] * abar ** k * bbar) for k in range(L)])
        want = np.array([sum(dy[0, d, t] * K[t - s] for t in range(s, L)) for s in range(L)])
        want += float(D[d]) * dy[0, d]
        assert _rel(g["du"][0, d], want) < 1e-12, (d, _rel(g["du"][0, d], want))


def test_bf16_storage_gradients_equal_widened_fp32():
    """The gradient oracle reads bf16 storage by exact widening: bf16 inputs give the gradients of
    the same values stored as fp32."""
    import synth
    c, dy, ds, softplus = _case(31, L=12)
    c16 = {k: (None if v is None or k in ("A", "D", "delta_bias", "h0") else synth.f32_to_bf16_bits(v))
           for k, v in c.items()}
    for k in ("A", "D", "delta_bias", "h0"):
        c16[k] = c[k]
    c32 = {k: (synth.bf16_bits_to_f32(v) if k not in ("A", "D", "delta_bias", "h0") and v is not None else v)
           for k, v in c16.items()}
    # one thread: the sums over channels then run in the same order in both calls
    a = oracle.scan_bwd(c16["u"], c16["delta"], c["A"], c16["B"], c16["C"], dy, c["D"], c16["z"],
                        c["delta_bias"], softplus, "bf16", h0=c["h0"], dlast_state=ds, nthreads=1)
    b = oracle.scan_bwd(c32["u"], c32["delta"], c["A"], c32["B"], c32["C"], dy, c["D"], c32["z"],
                        c["delta_bias"], softplus, "f32", h0=c["h0"], dlast_state=ds, nthreads=1)
    for k in a:
        if a[k] is not None:
            np.testing.assert_array_equal(a[k], b[k])


def test_bwd_f64_inputs_match_fp32():
    """Gradient oracle with inputs given as doubles: on fp32-representable values it equals the fp32
    run (single-threaded, so the sums over channels run in the same order), and an input perturbed
    below fp32 resolution changes the result (the doubles are not rounded)."""
    cfg = synth.CONFIGS["m130"].replace(batch=2, dim=5, seqlen=30, seed=4)
    inp = synth.scan_inputs(cfg)
    g = synth.grad_inputs(cfg)
    w = {k: inp[k].astype(np.float64) for k in ("u", "delta", "B", "C", "z")}
    dy = g["dy"].astype(np.float64)
    args = dict(h0=g["h0"], dlast_state=g["dlast"], nthreads=1)
    r32 = oracle.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], dy, inp["D"], inp["z"],
                          inp["delta_bias"], True, "f32", **args)
    r64 = oracle.scan_bwd(w["u"], w["delta"], inp["A"], w["B"], w["C"], dy, inp["D"], w["z"],
                          inp["delta_bias"], True, "f64", **args)
    for k in ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0"):
        assert np.array_equal(r32[k], r64[k]), k
    u2 = w["u"].copy()
    u2[0, 0, 0] += 1e-12
    r2 = oracle.scan_bwd(u2, w["delta"], inp["A"], w["B"], w["C"], dy, inp["D"], w["z"], inp["delta_bias"], True,
                         "f64", **args)
    assert not np.array_equal(r2["dB"], r64["dB"])
