"""Parity of the entropy-confidence variant (dspark_score_entropy) with the oracle.

"SGLang Integrates DSpark ...", "DSpark's Core Idea: Only Verify the Parts
You're Confident About": conf = exp(-H(softmax(z_q / theta))) of each draft
row, then the survival curve, budget, cap and scans of the head path, then
packing and verify as usual.  conf and S within 5e-5 absolute (conf also
2e-4 relative); every integer output exact apart from flagged near ties.
theta = 0.3 puts the synthetic drafts' confidences across (0, 1) (median
~0.26 on the mixed workload), so budgets span 0..gamma.
"""
import numpy as np
import pytest

from confidence_driven_speculative_gb300 import workloads as W
from tests.gpu_harness import compare_with_oracle, gpu_step, to_device

pytestmark = pytest.mark.gpu


def run_and_compare(inp_cpu, theta, **kw):
    gpu, bufs = gpu_step(to_device(inp_cpu), entropy_theta=theta)
    stats = compare_with_oracle(W.to_numpy(inp_cpu), gpu, entropy_theta=theta, **kw)
    return gpu, stats


@pytest.mark.parametrize("Tm", [0.0, 1.0])
@pytest.mark.parametrize("theta", [0.2, 0.5, 1.0])
def test_tiny_workload(cuda_lib, Tm, theta):
    for step in range(2):
        inp = W.make_inputs(W.TINY, step, temperature=Tm, cost_c=0.02)
        run_and_compare(inp, theta)


SHAPES = [  # B, gamma, V, d, dtype
    (1, 1, 8, 8, "bf16"),
    (3, 5, 8200, 40, "bf16"),      # 2 tiles, the second 16 bytes
    (37, 7, 20000, 264, "bf16"),   # 3 tiles, ragged
    (5, 16, 12292, 100, "f32"),    # 4 fp32 tiles, ragged
    (300, 4, 520, 64, "bf16"),     # many requests, one tile each
    (9, 64, 1000, 16, "bf16"),     # the largest gamma
]


@pytest.mark.parametrize("shape", SHAPES)
def test_small_shapes(cuda_lib, shape):
    B, g, V, d, dt = shape
    base = W.TINY if dt == "f32" else W.MIXED_B256
    for step, (T, c) in enumerate([(-1, 0.05), (max(1, B * g // 3), 0.001)]):
        inp = W.make_inputs(base, 30 + step, B=B, gamma=g, V=V, d=d, temperature=0.8,
                            cap_T=T, cost_c=c)
        run_and_compare(inp, 0.3)


def test_cost_edges(cuda_lib):
    for c in (-0.5, 0.0, 1.0, 1.5):
        inp = W.make_inputs(W.MIXED_B256, 7, B=8, V=4096, d=16, cap_T=-1, cost_c=c)
        gpu, _ = run_and_compare(inp, 0.3)
        if c <= 0:
            assert np.all(gpu["L"] == inp["gamma"])
        if c > 1:
            assert np.all(gpu["L"] == 0)


def test_masked_ids_do_not_count(cuda_lib):
    """-inf logits (masked ids) carry no probability: the row's entropy is
    that of its finite part.  Score step only (the verify takes finite
    logits)."""
    import oracle
    from confidence_driven_speculative_gb300 import binding
    from tests.gpu_harness import EPS_S_ENT, RTOL_CONF_ENT, TOL_S_ENT
    inp = W.make_inputs(W.MIXED_B256, 8, B=4, V=8192, d=16, cap_T=-1, cost_c=0.01)
    inp["draft_logits"][:, :, 100:3000] = float("-inf")
    inp["draft_logits"][0, 0, :4096] = float("-inf")   # a whole first half masked
    dev = to_device(inp)
    bufs = binding.StepBuffers(inp["B"], inp["gamma"], inp["V"], inp["d"])
    bufs.bind(dev)
    binding.dspark_score_entropy(bufs.step, 0.3)
    conf_g = bufs.conf.cpu().numpy()
    surv_g = bufs.survival.cpu().numpy()
    L0_g = bufs.L0.cpu().numpy()
    assert bufs.device_status() == 0
    conf, surv, L0, tie = oracle.score_entropy(W.to_numpy(inp)["draft_logits"], 0.3, 0.01,
                                               EPS_S_ENT)
    np.testing.assert_allclose(conf_g, conf, rtol=RTOL_CONF_ENT, atol=1e-12)
    np.testing.assert_allclose(surv_g, surv, rtol=0, atol=TOL_S_ENT)
    assert np.array_equal(L0_g[tie == 0], L0[tie == 0])


def test_latency_b1(cuda_lib):
    run_and_compare(W.make_inputs(W.LATENCY_B1, 0), 0.3)


@pytest.mark.slow
def test_mixed_b256(cuda_lib):
    gpu, stats = run_and_compare(W.make_inputs(W.MIXED_B256, 0), 0.3)
    assert 0 < gpu["L"].sum() <= 768
