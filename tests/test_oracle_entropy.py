"""Pins for the oracle's entropy-confidence variant.

Source: "SGLang Integrates DSpark ...", section "DSpark's Core Idea: Only
Verify the Parts You're Confident About": a draft position whose output
distribution has low entropy is a confident one.  Reading pinned here:
conf = exp(-H(softmax(z_q / theta))), then the survival curve and budget of
"DFlash to DSpark in SGLang", "DSpark: a sequential head and a verify
budget".

The pins come from outside the oracle's own loops: closed forms (uniform and
two-level rows), ``scipy.stats.entropy`` on the library softmax, the
invariances of the entropy (shift, permutation), its limits in theta, exact
bf16 widening, and the budget definition checked by brute force.
"""
import numpy as np
import pytest
from scipy import special, stats

import oracle


def _bf16_bits(x):
    """Round-to-nearest-even fp32 -> bf16 bit patterns (uint16)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def test_uniform_row_has_conf_one_over_V():
    for V in (1, 2, 7, 1000):
        z = np.full((1, 1, V), 3.25, np.float32)
        conf, _, _, _ = oracle.score_entropy(z, 1.0, 0.5)
        np.testing.assert_allclose(conf[0, 0], 1.0 / V, rtol=1e-12)


@pytest.mark.parametrize("k,V,a", [(1, 10, 2.0), (3, 50, 1.5), (5, 5, 0.0), (2, 1000, 7.0)])
def test_two_level_row_closed_form(k, V, a):
    # k tokens at logit a, V - k at 0: with Z = k e^a + V - k,
    # H = ln Z - k a e^a / Z.
    z = np.zeros((1, 1, V), np.float32)
    z[0, 0, :k] = a
    Z = k * np.exp(a) + (V - k)
    H = np.log(Z) - k * a * np.exp(a) / Z
    conf, _, _, _ = oracle.score_entropy(z, 1.0, 0.5)
    np.testing.assert_allclose(conf[0, 0], np.exp(-H), rtol=1e-12)


@pytest.mark.parametrize("theta", [0.5, 1.0, 2.0])
def test_matches_scipy_entropy_of_the_library_softmax(theta):
    rng = np.random.default_rng(3)
    B, g, V = 3, 4, 257
    z = (rng.normal(0, 2.0, (B, g, V))).astype(np.float32)
    th = float(np.float32(theta))
    conf, _, _, _ = oracle.score_entropy(z, theta, 0.5)
    for b in range(B):
        for i in range(g):
            q = special.softmax(z[b, i].astype(np.float64) / th)
            np.testing.assert_allclose(conf[b, i], np.exp(-stats.entropy(q)), rtol=1e-10)


def test_shift_and_permutation_invariance_and_one_hot_limit():
    rng = np.random.default_rng(4)
    z = rng.normal(0, 1.0, (2, 3, 64)).astype(np.float32)
    c0, _, _, _ = oracle.score_entropy(z, 1.0, 0.5)
    c1, _, _, _ = oracle.score_entropy(z + np.float32(4.0), 1.0, 0.5)
    np.testing.assert_allclose(c1, c0, rtol=1e-6)
    perm = rng.permutation(64)
    c2, _, _, _ = oracle.score_entropy(z[..., perm], 1.0, 0.5)
    np.testing.assert_allclose(c2, c0, rtol=1e-12)
    # theta -> 0: q tends to the one-hot of the unique maximum, conf -> 1;
    # theta -> infinity: q tends to uniform, conf -> 1/V
    c_cold, _, _, _ = oracle.score_entropy(z, 1e-4, 0.5)
    assert np.all(c_cold > 1 - 1e-6)
    c_hot, _, _, _ = oracle.score_entropy(z, 1e6, 0.5)
    np.testing.assert_allclose(c_hot, 1 / 64, rtol=1e-4)
    # sharper rows are more confident
    c_sharp, _, _, _ = oracle.score_entropy(z * np.float32(3), 1.0, 0.5)
    assert np.all(c_sharp > c0)


def test_bf16_rows_are_widened_exactly():
    rng = np.random.default_rng(5)
    z = rng.normal(0, 2.0, (2, 2, 300)).astype(np.float32)
    bits = _bf16_bits(z)
    widened = (bits.astype(np.uint32) << 16).view(np.float32)
    c_bf, s_bf, l_bf, _ = oracle.score_entropy(bits, 0.7, 0.01)
    c_f, s_f, l_f, _ = oracle.score_entropy(widened, 0.7, 0.01)
    np.testing.assert_array_equal(c_bf, c_f)
    np.testing.assert_array_equal(l_bf, l_f)


@pytest.mark.parametrize("c", [0.0, 0.02, 0.2, 0.6, 1.0, 1.5])
def test_survival_and_budget_definition(c):
    rng = np.random.default_rng(6)
    B, g, V = 6, 9, 40
    z = (rng.normal(0, 1.0, (B, g, V)) * rng.uniform(0.5, 6.0, (B, g, 1))).astype(np.float32)
    conf, surv, L0, tie = oracle.score_entropy(z, 1.0, c)
    assert np.all((conf > 1.0 / V - 1e-15) & (conf <= 1.0))
    np.testing.assert_allclose(surv, np.cumprod(conf, axis=1), rtol=1e-14)
    cf = float(np.float32(c))
    Sx = np.concatenate([np.ones((B, 1)), surv], axis=1)
    for b in range(B):
        ks = [k for k in range(g + 1) if Sx[b, k] >= cf]
        assert L0[b] == (max(ks) if ks else 0)
    # a near tie is any S_k (k = 0..gamma) within eps of c
    expect = (np.abs(Sx - cf) < 1e-5).sum(axis=1)
    np.testing.assert_array_equal(tie, expect)


def test_budget_counts_a_gain_equal_to_the_cost():
    # a uniform row over V = 2 ids has conf = 1/2 exactly, so S_k = 2^-k is
    # exact; L0 = max{k : S_k >= c} includes S_k == c
    z = np.zeros((1, 3, 2), np.float32)
    for c, L0_expect in [(0.5, 1), (0.25, 2), (0.125, 3), (0.2, 2)]:
        conf, surv, L0, tie = oracle.score_entropy(z, 1.0, c)
        np.testing.assert_array_equal(surv[0], [0.5, 0.25, 0.125])
        assert L0[0] == L0_expect, c
