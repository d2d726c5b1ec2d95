"""Parity of the cap-accept audit arm (dspark_verify_cap_accept) with the oracle.

"DFlash to DSpark in SGLang", "The confidence scheduler and verify modes":
the full block is verified (static layout, every L_b = gamma) and the
scheduler's window W_b is committed.  The window comes from the oracle's
own budget rule on the same inputs, or from a seeded draw that also covers
out-of-range values (the library clamps W_b to [0, L_b]).

Checked exactly: the full-block acceptance a_b, the committed accept
lengths, emitted tokens and cached lengths, and the batch totals; p(d) and
q(d) of every draft of the block within 1e-3 relative.  Requests the oracle
flags as a near tie are checked for validity only.
"""
import numpy as np
import pytest
import torch

import oracle
from confidence_driven_speculative_gb300 import binding
from confidence_driven_speculative_gb300 import workloads as W
from tests.gpu_harness import EPS_CAP, EPS_S, EPS_U, RTOL_P, to_device

pytestmark = pytest.mark.gpu


def scheduler_window(inp_np):
    """The window the confidence scheduler gives this step (oracle's rule)."""
    _, surv, L0, _ = oracle.score(inp_np["hidden"], inp_np["head_w"], inp_np["head_bias"],
                                  inp_np["sts_tau"], inp_np["cost_c"], EPS_S)
    L, _ = oracle.cap(surv, L0, inp_np["cap_T"], EPS_CAP)
    return L.astype(np.int32)


def gpu_cap_accept(inp_dev, window, L=None):
    """The audited block is static (every L_b = gamma) unless ``L`` gives
    the layout explicitly (offsets by torch cumsum, packing by the library)."""
    B, g, V, d = inp_dev["B"], inp_dev["gamma"], inp_dev["V"], inp_dev["d"]
    bufs = binding.StepBuffers(B, g, V, d)
    commit = inp_dev["seq_lens"].clone()
    bufs.bind(inp_dev, seq_lens_commit=commit)
    if L is None:
        bufs.step.cap_T = binding.DSPARK_NO_CAP
        bufs.step.fixed_budget = g                  # the audited block: static
        binding.dspark_score_budget(bufs.step)
    else:
        Lt = torch.as_tensor(np.asarray(L, np.int32)).cuda()
        z = torch.zeros(1, dtype=torch.int32, device="cuda")
        bufs.L.copy_(Lt)
        bufs.draft_off.copy_(torch.cat([z, torch.cumsum(Lt, 0).to(torch.int32)]))
        bufs.row_off.copy_(torch.cat([z, torch.cumsum(Lt + 1, 0).to(torch.int32)]))
    binding.dspark_compact(bufs.step)
    torch.cuda.synchronize()
    n_rows = int(bufs.row_off[B].item())
    tgt = W.ragged_target_rows(inp_dev["target_dense"], bufs.row_req, bufs.row_k,
                               n_rows).contiguous()
    bufs.bind_target(tgt)
    win = torch.as_tensor(window, dtype=torch.int32).cuda()
    accept_full = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    totals = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    binding.dspark_verify_cap_accept(bufs.step, win, accept_full, totals)
    torch.cuda.synchronize()
    assert bufs.device_status() == 0
    out = {k: getattr(bufs, k).cpu().numpy() for k in (
        "L", "accept_len", "num_emitted", "out_tokens", "p_tok", "q_tok")}
    out["accept_full"] = accept_full.cpu().numpy()
    out["audit_totals"] = totals.cpu().numpy()
    out["seq_lens_commit"] = commit.cpu().numpy()
    return out, bufs


def run_and_compare(inp_cpu, window, max_flag_frac=0.05, L=None):
    inp = W.to_numpy(inp_cpu)
    B, g = inp["draft_tokens"].shape
    gpu, bufs = gpu_cap_accept(to_device(inp_cpu), window, L)
    L = np.full(B, g, np.int32) if L is None else np.asarray(L, np.int32)
    assert np.array_equal(gpu["L"], L)
    ora = oracle.verify_cap_accept(inp["draft_tokens"], inp["draft_logits"], inp["target_dense"],
                                   L, window, inp["temperature"], inp["seed"], EPS_U,
                                   inp["seq_lens"])
    flagged = ora["tie"] > 0
    assert flagged.sum() <= max(3, int(max_flag_frac * B))
    ok = ~flagged
    for k in ("accept_full", "accept_len", "num_emitted", "out_tokens"):
        assert np.array_equal(gpu[k][ok], ora[k][ok]), k
    assert np.array_equal(gpu["seq_lens_commit"][ok], ora["seq_lens"][ok])
    Wc = ora["W"]
    assert np.array_equal(gpu["accept_len"], np.minimum(gpu["accept_full"], Wc))
    assert gpu["audit_totals"].tolist() == [int(gpu["accept_full"].sum()),
                                            int(gpu["accept_len"].sum())]
    if not flagged.any():
        assert gpu["audit_totals"].tolist() == ora["audit_totals"].tolist()
    if inp["temperature"] > 0:
        n = int(L.sum())
        np.testing.assert_allclose(gpu["p_tok"][:n].astype(np.float64), ora["p_tok"],
                                   rtol=RTOL_P, atol=1e-30)
        np.testing.assert_allclose(gpu["q_tok"][:n].astype(np.float64), ora["q_tok"],
                                   rtol=RTOL_P, atol=1e-30)
    # A flagged request: only decisions inside their tolerance window may go
    # the GPU's way.  The full verify fixes accept_full; the committed outcome
    # is the window verify's (window min(W, L)).
    for b in np.nonzero(flagged)[0]:
        a_full, a = int(gpu["accept_full"][b]), int(gpu["accept_len"][b])
        Lb, Wb = int(L[b]), int(Wc[b])
        un = np.array([oracle.uniforms(inp["seed"], int(b), k) for k in range(Lb + 1)])
        tgt_b = inp["target_dense"][b]
        dft_b = inp["draft_logits"][b]
        drafts = inp["draft_tokens"][b]
        v_full, _ = oracle.check_request(Lb, drafts[:max(Lb, 1)], tgt_b[:Lb + 1], dft_b[:max(Lb, 1)],
                                         inp["temperature"], un[:, 0], un[:, 1], un[:, 2],
                                         a_full, -1, eps=EPS_U)
        assert v_full == 0, (int(b), v_full, a_full)
        assert np.array_equal(gpu["out_tokens"][b, :a], drafts[:a])
        assert np.all(gpu["out_tokens"][b, a + 1:] == -1)
        v_win, _ = oracle.check_request(Wb, drafts[:max(Wb, 1)], tgt_b[:Wb + 1], dft_b[:max(Wb, 1)],
                                        inp["temperature"], un[:Wb + 1, 0], un[:Wb + 1, 1],
                                        un[:Wb + 1, 2], a, int(gpu["out_tokens"][b, a]), eps=EPS_U)
        assert v_win == 0, (int(b), v_win, a)
    return gpu, ora, bufs


@pytest.mark.parametrize("Tm", [0.0, 1.0])
def test_tiny_scheduler_window(cuda_lib, Tm):
    for step in range(3):
        inp = W.make_inputs(W.TINY, step, temperature=Tm)
        run_and_compare(inp, scheduler_window(W.to_numpy(inp)))


SHAPES = [  # B, gamma, V, d, dtype
    (3, 5, 8200, 40, "bf16"),      # 2 tiles, the second 16 bytes
    (37, 7, 20000, 264, "bf16"),   # 3 tiles, ragged
    (5, 16, 12292, 100, "f32"),    # 4 fp32 tiles, ragged
    (300, 4, 520, 64, "bf16"),     # many requests, one tile each
    (9, 64, 1000, 16, "bf16"),     # the largest gamma
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("Tm", [0.0, 0.8])
def test_small_shapes_random_windows(cuda_lib, shape, Tm):
    B, g, V, d, dt = shape
    base = W.TINY if dt == "f32" else W.MIXED_B256
    inp = W.make_inputs(base, 20, B=B, gamma=g, V=V, d=d, temperature=Tm, cap_T=-1, cost_c=0.0)
    rng = np.random.default_rng(1000 + B + g)
    window = rng.integers(-2, g + 3, B).astype(np.int32)   # includes W < 0 and W > gamma
    window[0] = 0
    window[-1] = g
    run_and_compare(inp, window)


def test_window_inside_the_accepted_run(cuda_lib):
    """Draft logits equal to the target's: every draft is accepted, so every
    window shorter than the block ends inside the accepted run and its token
    is drawn from p at row W_b."""
    inp = W.make_inputs(W.MIXED_B256, 3, B=24, V=20000, d=64, cap_T=-1, cost_c=0.0)
    inp["draft_logits"] = inp["target_dense"][:, :-1].clone()
    g = inp["gamma"]
    window = (np.arange(24) % (g + 1)).astype(np.int32)
    gpu, _, _ = run_and_compare(inp, window)
    assert np.all(gpu["accept_full"] == g)
    assert np.array_equal(gpu["accept_len"], window)


def test_window_covering_the_block_is_the_static_verify(cuda_lib):
    inp = W.make_inputs(W.MIXED_B256, 5, B=16, V=20000, d=64, cap_T=-1, cost_c=0.0)
    g = inp["gamma"]
    gpu, _, _ = run_and_compare(inp, np.full(16, g, np.int32))
    assert np.array_equal(gpu["accept_len"], gpu["accept_full"])
    # the same block through dspark_verify (at B = 16 its small-batch path,
    # which sums the softmax in another order: p and q agree to rounding)
    from tests.gpu_harness import gpu_step
    inp_s = dict(inp, fixed_budget=g)
    st, _ = gpu_step(to_device(inp_s))
    for k in ("accept_len", "num_emitted", "out_tokens"):
        assert np.array_equal(st[k], gpu[k]), k
    for k in ("p_tok", "q_tok"):
        np.testing.assert_allclose(st[k], gpu[k], rtol=1e-5, atol=1e-30)


def test_latency_b1_scheduler_window(cuda_lib):
    inp = W.make_inputs(W.LATENCY_B1, 0)
    run_and_compare(inp, scheduler_window(W.to_numpy(inp)))


@pytest.mark.slow
def test_mixed_b256_scheduler_window(cuda_lib):
    inp = W.make_inputs(W.MIXED_B256, 0)
    gpu, ora, _ = run_and_compare(inp, scheduler_window(W.to_numpy(inp)))
    tot = gpu["audit_totals"]
    assert 0 < tot[1] <= tot[0]


@pytest.mark.parametrize("Tm", [0.0, 1.0])
def test_layout_with_empty_requests(cuda_lib, Tm):
    """A verified block with L_b = 0 for some requests (only their bonus row
    is read): a_b = 0 there, and every other output as the oracle's."""
    B, g, V, d = 24, 6, 8200, 40
    inp = W.make_inputs(W.MIXED_B256, 21, B=B, gamma=g, V=V, d=d, temperature=Tm,
                        cap_T=-1, cost_c=0.0)
    rng = np.random.default_rng(77)
    L = rng.integers(0, g + 1, B).astype(np.int32)
    L[:4] = 0
    window = rng.integers(-1, g + 2, B).astype(np.int32)
    gpu, ora, _ = run_and_compare(inp, window, L=L)
    assert np.all(gpu["accept_full"][:4] == 0)
    assert np.all(gpu["accept_full"] <= L)
