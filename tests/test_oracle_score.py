"""Pins for the oracle's confidence head, survival curve and budget rule.

Source: "DFlash to DSpark in SGLang", section "DSpark: a sequential head and a
verify budget" (linear + sigmoid head, survival = product of scores, STS) and
section "The confidence scheduler and verify modes" (walk down the curve, stop
at the marginal cost).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def _rand_inputs(B=5, gamma=7, d=33, seed=0, bias=0.5, dtype=np.float32):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((B, gamma, d)).astype(np.float32)
    w = (rng.standard_normal(d) / math.sqrt(d)).astype(np.float32)
    b = np.full(B, bias, np.float32)
    tau = (1.0 + 0.05 * np.arange(gamma)).astype(np.float32)
    return h, w, b, tau


def test_worked_example():
    g = GOLDEN["score"]
    h = np.array(g["hidden"], np.float32).reshape(1, 4, 1)
    w = np.ones(1, np.float32)
    tau = np.array(g["tau"], np.float32)
    for case in g["cases"]:
        conf, surv, L0, _ = oracle.score(h, w, np.zeros(1, np.float32), tau, case["c"])
        np.testing.assert_allclose(conf[0], g["conf"], atol=1e-6)
        np.testing.assert_allclose(surv[0], g["surv"], atol=1e-6)
        assert L0[0] == case["L0"], case


def test_large_bias_gives_certain_drafts():
    h, w, _, tau = _rand_inputs()
    conf, surv, L0, _ = oracle.score(h, w, np.full(5, 1e4, np.float32), tau, 0.999)
    assert np.all(conf == 1.0) and np.all(surv == 1.0) and np.all(L0 == 7)


def test_infinite_temperature_gives_one_half():
    h, w, b, _ = _rand_inputs()
    tau = np.full(7, 1e30, np.float32)
    conf, surv, L0, _ = oracle.score(h, w, b, tau, 0.1)
    np.testing.assert_allclose(conf, 0.5, atol=1e-12)
    np.testing.assert_allclose(surv, np.broadcast_to(0.5 ** np.arange(1, 8), surv.shape), rtol=1e-12)
    # S_k = 2^-k >= 0.1 for k <= 3
    assert np.all(L0 == 3)


def test_sigmoid_symmetry_and_linearity_of_the_logit():
    """logit(conf) * tau - bias must be a linear function of h (the projection
    w.h): additive in h, zero at h = 0, and flipping h and bias flips conf."""
    h1, w, b, tau = _rand_inputs(seed=1, bias=0.3)
    h2, _, _, _ = _rand_inputs(seed=2)
    def proj(h, bias):
        conf, _, _, _ = oracle.score(h, w, bias, tau, 0.5)
        return np.log(conf / (1 - conf)) * tau[None, :] - bias[:, None]
    p1, p2, p12 = proj(h1, b), proj(h2, b), proj(h1 + h2, b)
    np.testing.assert_allclose(p12, p1 + p2, atol=2e-5)
    np.testing.assert_allclose(proj(np.zeros_like(h1), b), 0.0, atol=1e-9)
    c1, _, _, _ = oracle.score(h1, w, b, tau, 0.5)
    c2, _, _, _ = oracle.score(-h1, w, -b, tau, 0.5)
    np.testing.assert_allclose(c1 + c2, 1.0, atol=1e-12)


def test_projection_uses_every_coordinate():
    """A one-hot hidden state picks out one weight: logit = (w_j + b) / tau."""
    d, gamma = 9, 3
    w = np.linspace(-1, 1, d).astype(np.float32)
    tau = np.array([1.0, 2.0, 4.0], np.float32)
    for j in range(d):
        h = np.zeros((1, gamma, d), np.float32)
        h[0, :, j] = 1.0
        conf, _, _, _ = oracle.score(h, w, np.array([0.25], np.float32), tau, 0.5)
        logit = np.log(conf[0] / (1 - conf[0]))
        np.testing.assert_allclose(logit * tau, float(w[j]) + 0.25, atol=1e-9)


@pytest.mark.parametrize("c", [-0.5, 0.0, 0.2, 0.5, 0.9, 1.0, 1.2])
def test_survival_invariants_and_budget_definition(c):
    h, w, b, tau = _rand_inputs(B=20, gamma=16, d=64, seed=3, bias=1.0)
    conf, surv, L0, _ = oracle.score(h, w, b, tau, c)
    assert np.all((conf >= 0) & (conf <= 1))
    assert np.all((surv >= 0) & (surv <= 1))
    assert np.all(np.diff(surv, axis=1) <= 0)          # monotone non-increasing
    np.testing.assert_allclose(surv[:, 0], conf[:, 0], rtol=1e-15)
    np.testing.assert_allclose(surv[:, 1:], surv[:, :-1] * conf[:, 1:], rtol=1e-14)
    assert np.all((L0 >= 0) & (L0 <= 16))
    S = np.concatenate([np.ones((20, 1)), surv], axis=1)  # S_0 .. S_gamma
    for bb in range(20):
        if c > 1:
            assert L0[bb] == 0
        else:
            assert S[bb, L0[bb]] >= c
            assert L0[bb] == 16 or S[bb, L0[bb] + 1] < c
    if c <= 0:
        assert np.all(L0 == 16)


def test_bf16_hidden_is_widened_exactly():
    h, w, b, tau = _rand_inputs(seed=4)
    bits = (h.view(np.uint32) >> 16).astype(np.uint16)      # truncate to bf16
    widened = (bits.astype(np.uint32) << 16).view(np.float32)
    c1, s1, l1, _ = oracle.score(bits, w, b, tau, 0.4)
    c2, s2, l2, _ = oracle.score(widened, w, b, tau, 0.4)
    np.testing.assert_array_equal(c1, c2)
    np.testing.assert_array_equal(l1, l2)


def test_near_tie_flag():
    h = np.zeros((1, 2, 1), np.float32)
    w = np.ones(1, np.float32)
    tau = np.ones(2, np.float32)
    # conf = 0.5 each: S = [0.5, 0.25]; c exactly at S_2 is a near tie
    _, _, L0, tie = oracle.score(h, w, np.zeros(1, np.float32), tau, 0.25, eps=1e-5)
    assert L0[0] == 2 and tie[0] == 1
    _, _, _, tie = oracle.score(h, w, np.zeros(1, np.float32), tau, 0.3, eps=1e-5)
    assert tie[0] == 0
