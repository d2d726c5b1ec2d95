"""Parity of the STS temperature fit (dspark_fit_sts_tau) with the oracle.

"DFlash to DSpark in SGLang", "DSpark: a sequential head and a verify
budget": STS calibrates the survival product to true acceptance.  Both
sides fit the maximum-likelihood temperature per position on the same logs;
the oracle by golden-section search on the likelihood in fp64, the kernel by
bisection on its derivative (fp32 terms, fp64 sums).  Observation counts are
exact; tau agrees within 1e-4 relative (both sides resolve the convex
optimum far more finely: the kernel's fp32 terms move the root by ~1e-6
relative at these sizes, the oracle's search stops at ~1e-8); the
likelihood at the optimum within 1e-5 relative.

Logs are synthetic (a ground-truth temperature per position draws the
outcomes) or come from the oracle's own step on the tiny workload; none
comes from the CUDA path.
"""
import numpy as np
import pytest
import torch
from scipy import special

import oracle
from confidence_driven_speculative_gb300 import binding
from confidence_driven_speculative_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def synthetic_logs(seed, N, g, tau_lo=0.5, tau_hi=3.0, x_mean=1.0, full=False):
    """Logs drawn from a known temperature per position: head logits x,
    outcomes accept ~ sigmoid(x / tau_true), a = first rejection, verify
    lengths L uniform in 0..g (or all g), a cut at L."""
    rng = np.random.default_rng(seed)
    tau_true = rng.uniform(tau_lo, tau_hi, g)
    tau_used = rng.uniform(0.5, 2.0, g).astype(np.float32)
    x = rng.normal(x_mean, 2.0, (N, g))
    acc = rng.random((N, g)) < special.expit(x / tau_true)
    a = np.where(acc.all(axis=1), g, np.argmin(acc, axis=1)).astype(np.int32)
    L = rng.integers(0, g + 1, N).astype(np.int32)
    if full:
        L[:] = g
    a = np.minimum(a, L)
    conf = special.expit(x / tau_used).astype(np.float32)
    return conf, tau_used, L, a, tau_true


def fit_both(conf, tau_used, L, a, tau_min=0.05, tau_max=20.0):
    g = conf.shape[1]
    dev = lambda v: torch.as_tensor(np.ascontiguousarray(v)).cuda()
    tau = torch.full((g,), -1.0, dtype=torch.float32, device="cuda")
    nll = torch.full((g,), -1.0, dtype=torch.float32, device="cuda")
    nobs = torch.full((g,), -1, dtype=torch.int32, device="cuda")
    binding.dspark_fit_sts_tau(dev(conf), dev(tau_used), dev(L), dev(a), tau, tau_min, tau_max,
                               nll_out=nll, n_obs=nobs)
    torch.cuda.synchronize()
    t_o, n_o, c_o = oracle.fit_sts_tau(conf, tau_used, L, a, tau_min, tau_max)
    t_g, n_g, c_g = tau.cpu().numpy(), nll.cpu().numpy(), nobs.cpu().numpy()
    assert np.array_equal(c_g, c_o)
    np.testing.assert_allclose(t_g, t_o, rtol=1e-4)
    np.testing.assert_allclose(n_g, n_o, rtol=1e-5, atol=1e-6)
    return t_g, t_o, c_o


@pytest.mark.parametrize("seed,N,g", [(0, 400, 6), (1, 5000, 16), (2, 60000, 16), (3, 37, 64)])
def test_synthetic_logs(cuda_lib, seed, N, g):
    fit_both(*synthetic_logs(seed, N, g)[:4])


def test_recovers_the_generating_temperatures(cuda_lib):
    conf, tau_used, L, a, tau_true = synthetic_logs(5, 200000, 8, 0.7, 2.0, x_mean=3.0,
                                                    full=True)
    t_g, _, nobs = fit_both(conf, tau_used, L, a)
    # maximum likelihood is consistent: with >= 10^4 observations per position
    # the fit lands within a few percent of the generating temperature
    assert np.all(nobs > 10000)
    np.testing.assert_allclose(t_g, tau_true, rtol=0.05)


def test_bounds_and_empty_positions(cuda_lib):
    conf = np.full((5, 3), 0.9, np.float32)
    L = np.ones(5, np.int32)
    t, _, nobs = fit_both(conf, np.array([1.0, 1.5, 2.0], np.float32), L,
                          np.zeros(5, np.int32), 0.1, 10.0)
    assert nobs.tolist() == [5, 0, 0]
    assert t[0] == pytest.approx(10.0) and t[1:].tolist() == [1.5, 2.0]
    t, _, _ = fit_both(conf, np.array([1.0, 1.5, 2.0], np.float32), L, np.ones(5, np.int32),
                       0.1, 10.0)
    assert t[0] == pytest.approx(0.1, rel=1e-6)
    # no logs at all: every temperature unchanged
    t, _, nobs = fit_both(np.zeros((0, 4), np.float32), np.full(4, 1.25, np.float32),
                          np.zeros(0, np.int32), np.zeros(0, np.int32))
    assert nobs.tolist() == [0] * 4 and t.tolist() == [1.25] * 4


def test_logs_of_the_oracle_step(cuda_lib):
    """conf, L and accept lengths of the oracle's step on the tiny workload."""
    confs, Ls, accs = [], [], []
    for step in range(24):
        inp = W.to_numpy(W.make_inputs(W.TINY, step, cost_c=0.05, cap_T=-1))
        r = oracle.step(inp)
        confs.append(r["conf"].astype(np.float32))
        Ls.append(r["L"])
        accs.append(r["accept_len"])
    conf = np.concatenate(confs)
    fit_both(conf, W.to_numpy(W.make_inputs(W.TINY, 0))["sts_tau"].astype(np.float32),
             np.concatenate(Ls).astype(np.int32), np.concatenate(accs).astype(np.int32))
