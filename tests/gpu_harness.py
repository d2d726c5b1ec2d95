"""Helpers for the GPU parity tests: run the CUDA step through the C ABI and
compare it with the oracle, decision by decision.

Tolerances (from the fp32 arithmetic of the kernels against the fp64
oracle): conf and survival agree within TOL_S absolute; p(d), q(d) within
1e-3 relative (floor 1e-30).  Every
integer output is compared exactly, except a decision the oracle flags as a
near tie (its fp64 margin below the tolerance the fp32 kernels are held to).
There only that decision may go the GPU's way: a flagged budget or cap
boundary is checked valid and the oracle continues from the GPU's lengths;
in a flagged request every other accept test and draw must still match
(oracle.check_request).  The counts of open decisions are returned.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from confidence_driven_speculative_gb300 import binding, workloads

TOL_S = 1e-5           # |S_gpu - S_oracle|, |conf_gpu - conf_oracle|
EPS_S = 2 * TOL_S      # oracle near-tie window for S_k vs c
EPS_CAP = 4 * TOL_S    # oracle near-tie window between the T-th and (T+1)-th gains
EPS_U = 1e-5           # |u - min(1, p/q)| window named by the method's tolerance
RTOL_P = 1e-3
# Entropy confidence (conf = exp(-H)): the fp32 sums of 2^(y-m) and of
# 2^(y-m)(y-m) carry ~5e-6 relative error at worst after pairwise vector sums,
# which enters conf scaled by (1 + H) and S by the sum over k of (1 + H_k).
TOL_S_ENT = 5e-5
EPS_S_ENT = 2 * TOL_S_ENT
EPS_CAP_ENT = 4 * TOL_S_ENT
RTOL_CONF_ENT = 2e-4


def to_device(inp: dict, device="cuda") -> dict:
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def gpu_step(inp_dev: dict, seq_lens_commit: bool = True, bufs=None, stream=None,
             entropy_theta=None, fused: bool = False):
    """score_budget (or score_entropy) -> compact -> (target-forward
    stand-in) -> verify.  ``fused``: dspark_score_compact in place of the
    first two calls."""
    B, g, V, d = inp_dev["B"], inp_dev["gamma"], inp_dev["V"], inp_dev["d"]
    if bufs is None:
        bufs = binding.StepBuffers(B, g, V, d, stream=stream)
    commit = inp_dev["seq_lens"].clone() if seq_lens_commit else None
    bufs.bind(inp_dev, seq_lens_commit=commit)
    if fused:
        assert entropy_theta is None
        binding.dspark_score_compact(bufs.step, stream)
    else:
        if entropy_theta is None:
            binding.dspark_score_budget(bufs.step, stream)
        else:
            binding.dspark_score_entropy(bufs.step, entropy_theta, stream)
        binding.dspark_compact(bufs.step, stream)
    torch.cuda.synchronize()
    n_rows = int(bufs.row_off[B].item()) if B > 0 else 0
    tgt = workloads.ragged_target_rows(inp_dev["target_dense"], bufs.row_req, bufs.row_k,
                                       n_rows).contiguous()
    if tgt.numel() == 0:
        tgt = torch.zeros((1, V), dtype=inp_dev["target_dense"].dtype, device="cuda")
    bufs.bind_target(tgt)
    binding.dspark_verify(bufs.step, stream)
    torch.cuda.synchronize()
    assert bufs.device_status() == 0
    return outputs_of(bufs, commit), bufs


def outputs_of(bufs, commit=None) -> dict:
    """Host copies of every output a step wrote into ``bufs`` (the dict that
    ``compare_with_oracle`` takes)."""
    out = {k: getattr(bufs, k).cpu().numpy() for k in (
        "conf", "survival", "L0", "L", "draft_off", "row_off", "packed_ids", "packed_pos",
        "row_req", "row_k", "accept_len", "num_emitted", "out_tokens", "p_tok", "q_tok")}
    out["seq_lens_commit"] = commit.cpu().numpy() if commit is not None else None
    return out


def check_L_valid(S, c, L0, L, T, tol=TOL_S):
    """The GPU's L0 and L are a valid outcome of the budget rule and cap
    given fp64 survival S (B x gamma, S_1..S_gamma) and an fp32 error <= tol."""
    B, g = S.shape
    Sx = np.concatenate([np.ones((B, 1)), S], axis=1)
    for b in range(B):
        l0 = L0[b]
        assert 0 <= l0 <= g
        if l0 > 0:
            assert Sx[b, l0] >= c - tol, (b, l0)
        if l0 < g:
            assert not (Sx[b, l0 + 1] >= c + tol), (b, l0)
        if c > 1 + tol:
            assert l0 == 0
    assert np.all((L >= 0) & (L <= L0))
    if T < 0 or L0.sum() <= T:
        assert np.array_equal(L, L0)
        return
    assert L.sum() == T
    kept = [S[b, k] for b in range(B) for k in range(L[b])]
    dropped = [S[b, k] for b in range(B) for k in range(L[b], L0[b])]
    if kept and dropped:
        assert min(kept) >= max(dropped) - 2 * tol


def compare_with_oracle(inp_np: dict, gpu: dict, max_flag_frac: float = 0.05,
                        entropy_theta=None) -> dict:
    """Check every GPU output of one step against the oracle.  Returns counts.
    With ``entropy_theta`` the confidences are the entropy variant's."""
    B, g = inp_np["draft_tokens"].shape
    stats = {"score_ties": 0, "cap_tie": 0, "verify_ties": 0}
    fixed = inp_np.get("fixed_budget", -1)
    tol, eps_cap = (TOL_S, EPS_CAP) if entropy_theta is None else (TOL_S_ENT, EPS_CAP_ENT)
    if fixed is not None and fixed >= 0:
        L = oracle.fixed_budget(B, g, fixed)
        assert np.array_equal(gpu["L"], L)
    else:
        if entropy_theta is None:
            conf, surv, L0, tie = oracle.score(inp_np["hidden"], inp_np["head_w"],
                                               inp_np["head_bias"], inp_np["sts_tau"],
                                               inp_np["cost_c"], EPS_S)
        else:
            conf, surv, L0, tie = oracle.score_entropy(inp_np["draft_logits"], entropy_theta,
                                                       inp_np["cost_c"], EPS_S_ENT)
        np.testing.assert_allclose(gpu["conf"], conf, rtol=0, atol=tol)
        np.testing.assert_allclose(gpu["survival"], surv, rtol=0, atol=tol)
        if entropy_theta is not None:
            # relative error of exp(-H): (1 + H) times the sums' ~5e-6, H <= ln V
            np.testing.assert_allclose(gpu["conf"], conf, rtol=RTOL_CONF_ENT, atol=1e-12)
        assert np.all(np.diff(gpu["survival"], axis=1) <= 0)
        c = float(np.float32(inp_np["cost_c"]))
        untied = tie == 0
        assert np.array_equal(gpu["L0"][untied], L0[untied]), "pre-cap lengths differ"
        stats["score_ties"] = int((~untied).sum())
        # The GPU's lengths are a valid outcome of the budget and cap (this
        # covers the flagged near ties too).
        check_L_valid(surv, c, gpu["L0"], gpu["L"], inp_np["cap_T"], tol)
        # The oracle goes on from its own L0.  Only where it flagged a near
        # tie, where either choice is correct, does it take the GPU's (just
        # checked valid), so that the later stages compare like with like.
        L0_used = np.where(untied, L0, gpu["L0"]).astype(np.int32)
        Lcap, cap_tie = oracle.cap(surv, L0_used, inp_np["cap_T"], eps_cap)
        stats["cap_tie"] = cap_tie
        if cap_tie == 0:
            assert np.array_equal(gpu["L"], Lcap), "capped lengths differ"
            L = Lcap
        else:
            L = gpu["L"].astype(np.int32)  # a flagged cap boundary: the GPU's valid choice
    cpt = oracle.compact(L, inp_np["draft_tokens"], inp_np["last_tokens"], inp_np["seq_lens"])
    for k in ("draft_off", "row_off", "packed_ids", "packed_pos", "row_req", "row_k"):
        assert np.array_equal(gpu[k], cpt[k]), k
    tgt = oracle.ragged_target(inp_np["target_dense"], L, cpt["row_off"])
    ver = oracle.verify(inp_np["draft_tokens"], inp_np["draft_logits"], tgt, L, cpt["row_off"],
                        cpt["draft_off"], inp_np["temperature"], inp_np["seed"], EPS_U,
                        inp_np["seq_lens"])
    n = int(cpt["draft_off"][B])
    flagged = ver["tie"] > 0
    stats["verify_ties"] = int(flagged.sum())
    assert stats["verify_ties"] <= max(3, int(max_flag_frac * B)), stats
    ok = ~flagged
    assert np.array_equal(gpu["accept_len"][ok], ver["accept_len"][ok]), "accept lengths differ"
    assert np.array_equal(gpu["num_emitted"][ok], ver["num_emitted"][ok])
    assert np.array_equal(gpu["out_tokens"][ok], ver["out_tokens"][ok]), "emitted tokens differ"
    if inp_np["temperature"] > 0:
        p_o, q_o = ver["p_tok"], ver["q_tok"]
        p_g, q_g = gpu["p_tok"][:n].astype(np.float64), gpu["q_tok"][:n].astype(np.float64)
        np.testing.assert_allclose(p_g, p_o, rtol=RTOL_P, atol=1e-30)
        np.testing.assert_allclose(q_g, q_o, rtol=RTOL_P, atol=1e-30)
    # A flagged request: the oracle's decisions hold exactly except the ones
    # inside their tolerance window, where the GPU's side is taken; its
    # accept length and token must be such an outcome.
    kinds = np.zeros(3, np.int64)
    for b in np.nonzero(flagged)[0]:
        a = int(gpu["accept_len"][b])
        Lb = int(L[b])
        assert 0 <= a <= Lb
        assert np.array_equal(gpu["out_tokens"][b, :a], inp_np["draft_tokens"][b, :a])
        assert np.all(gpu["out_tokens"][b, a + 1:] == -1)
        assert gpu["num_emitted"][b] == a + 1
        r0 = int(cpt["row_off"][b])
        un = np.array([oracle.uniforms(inp_np["seed"], int(b), k) for k in range(Lb + 1)])
        verdict, kb = oracle.check_request(
            Lb, inp_np["draft_tokens"][b, :max(Lb, 1)], tgt[r0:r0 + Lb + 1],
            inp_np["draft_logits"][b, :max(Lb, 1)], inp_np["temperature"],
            un[:, 0], un[:, 1], un[:, 2], a, int(gpu["out_tokens"][b, a]), eps=EPS_U)
        assert verdict == 0, (int(b), verdict, a, int(gpu["out_tokens"][b, a]))
        kinds += kb
    stats["open_accept"], stats["open_zmass"], stats["open_draw"] = (int(x) for x in kinds)
    if gpu.get("seq_lens_commit") is not None:
        assert np.array_equal(gpu["seq_lens_commit"], inp_np["seq_lens"] + gpu["accept_len"] + 1)
    stats["mean_L"] = float(L.mean()) if B else 0.0
    stats["mean_accept"] = float(gpu["accept_len"].mean()) if B else 0.0
    return stats
