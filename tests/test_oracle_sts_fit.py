"""Pins for the oracle's STS temperature fit.

Source: "DFlash to DSpark in SGLang", section "DSpark: a sequential head and
a verify budget": Sequential Temperature Scaling calibrates the survival
product to match true acceptance rates.  Reading pinned here: per position,
the maximum-likelihood temperature of conf = sigmoid(x / tau) on the logged
outcomes, a position being observed when it was verified and every earlier
draft was accepted.

Pins: which positions a logged step observes (hand-worked), the closed form
for a constant logit (sigmoid(beta x) = accept fraction), agreement with
``scipy.optimize.minimize_scalar`` on the same likelihood, the bounds when
the data are separable, and the scaling of tau with the temperature that
produced the logged confidences.
"""
import numpy as np
import pytest
from scipy import optimize, special

import oracle


def _logit(p):
    return np.log(p) - np.log1p(-p)


def test_observed_positions_hand_worked():
    # step n: (L, a) -> observed positions and outcomes
    #   (3, 1): 0 accept, 1 reject            (2 is past the rejection)
    #   (3, 3): 0, 1, 2 accept                (nothing rejected)
    #   (2, 0): 0 reject
    #   (1, 1): 0 accept                      (1 was not verified)
    conf = np.full((4, 3), 0.7, np.float32)
    tau, nll, nobs = oracle.fit_sts_tau(conf, np.ones(3, np.float32), [3, 3, 2, 1], [1, 3, 0, 1])
    assert nobs.tolist() == [4, 2, 1]
    x = float(_logit(np.float64(np.float32(0.7))))
    # position 0: 3 accepts of 4 -> sigmoid(beta x) = 3/4 (golden-section on a
    # flat minimum resolves beta to ~sqrt(machine eps))
    np.testing.assert_allclose(tau[0], x / _logit(0.75), rtol=1e-6)
    # position 1: 1 of 2 -> beta = 0, clipped to the smallest beta (tau_max)
    assert tau[1] == pytest.approx(20.0)
    # position 2: all accepted with x > 0 -> the largest beta (tau_min)
    assert tau[2] == pytest.approx(np.float32(0.05), rel=1e-7)


@pytest.mark.parametrize("k,n,c,tu", [(7, 10, 2.0, 1.0), (2, 9, -1.3, 0.8), (40, 50, 0.6, 2.5)])
def test_constant_logit_closed_form(k, n, c, tu):
    # the logit and the accept fraction's logit share a sign, so beta > 0
    conf = np.full((n, 1), special.expit(c / tu), np.float32)
    a = np.array([1] * k + [0] * (n - k), np.int32)
    tau, nll, nobs = oracle.fit_sts_tau(conf, [tu], np.ones(n, np.int32), a)
    x = tu * _logit(np.float64(conf[0, 0]))
    assert nobs[0] == n
    np.testing.assert_allclose(tau[0], x / _logit(k / n), rtol=1e-6)
    p = k / n
    np.testing.assert_allclose(nll[0], -n * (p * np.log(p) + (1 - p) * np.log(1 - p)), rtol=1e-9)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_scipy_bounded_minimiser(seed):
    rng = np.random.default_rng(seed)
    N, g = 400, 6
    tau_true = rng.uniform(0.5, 3.0, g)
    tau_used = rng.uniform(0.5, 2.0, g).astype(np.float32)
    x = rng.normal(1.0, 2.0, (N, g))
    acc = rng.random((N, g)) < special.expit(x / tau_true)
    a = np.where(acc.all(axis=1), g, np.argmin(acc, axis=1)).astype(np.int32)
    L = rng.integers(1, g + 1, N).astype(np.int32)
    a = np.minimum(a, L)
    conf = special.expit(x / tau_used).astype(np.float32)
    tau, nll, nobs = oracle.fit_sts_tau(conf, tau_used, L, a, 0.05, 20.0)
    for i in range(g):
        obs = (i < L) & (i <= a)
        assert nobs[i] == obs.sum()
        xi = tau_used[i].astype(np.float64) * _logit(
            np.clip(conf[obs, i].astype(np.float64), 2.0 ** -126, 1 - 2.0 ** -24))
        yi = (i < a[obs]).astype(np.float64)

        def f(beta):
            return np.sum(np.logaddexp(0.0, beta * xi) - yi * beta * xi)

        r = optimize.minimize_scalar(f, bounds=(1 / 20.0, 1 / 0.05), method="bounded",
                                     options={"xatol": 1e-12})
        np.testing.assert_allclose(1 / tau[i], r.x, rtol=1e-5)
        assert nll[i] <= f(r.x) + 1e-9
        np.testing.assert_allclose(nll[i], f(1 / tau[i]), rtol=1e-12)


def test_separable_data_goes_to_the_bounds_and_empty_positions_keep_tau():
    conf = np.full((5, 3), 0.9, np.float32)   # x > 0 everywhere
    L = np.array([1, 1, 1, 1, 1], np.int32)
    tau, _, nobs = oracle.fit_sts_tau(conf, [1.0, 1.5, 2.0], L, np.zeros(5, np.int32), 0.1, 10.0)
    assert nobs.tolist() == [5, 0, 0]
    assert tau[0] == pytest.approx(10.0)          # every one rejected: smallest beta
    assert tau[1:].tolist() == [1.5, 2.0]         # no observation: unchanged
    tau, _, _ = oracle.fit_sts_tau(conf, [1.0, 1.5, 2.0], L, np.ones(5, np.int32), 0.1, 10.0)
    assert tau[0] == pytest.approx(np.float32(0.1), rel=1e-7)


def test_tau_scales_with_the_logging_temperature():
    rng = np.random.default_rng(9)
    N, g = 600, 4
    x = rng.normal(1.0, 2.0, (N, g))
    acc = rng.random((N, g)) < special.expit(x / 1.5)
    a = np.where(acc.all(axis=1), g, np.argmin(acc, axis=1)).astype(np.int32)
    L = np.full(N, g, np.int32)
    conf = special.expit(x).astype(np.float32)
    t1, _, _ = oracle.fit_sts_tau(conf, np.ones(g, np.float32), L, a, 0.01, 100.0)
    t2, _, _ = oracle.fit_sts_tau(conf, np.full(g, 2.0, np.float32), L, a, 0.01, 100.0)
    assert np.all((t1 > 0.02) & (t1 < 50))       # interior optima
    np.testing.assert_allclose(t2, 2 * t1, rtol=1e-6)
