"""The GPU parity harness, run on the CPU against the oracle's own outputs.

``compare_with_oracle`` must accept the oracle's step as a "GPU" result and
reject it once a single emitted token, length or probability is changed, so
that the GPU tests fail for the right reasons.
"""
import numpy as np
import pytest

import oracle
from confidence_driven_speculative_gb300 import workloads as W
from tests.gpu_harness import EPS_U, compare_with_oracle

KEYS = ("conf", "survival", "L0", "L", "draft_off", "row_off", "packed_ids", "packed_pos",
        "row_req", "row_k", "accept_len", "num_emitted", "out_tokens", "p_tok", "q_tok")


def oracle_as_gpu(inp):
    r = oracle.step(inp, eps_u=EPS_U)
    B, g_ = inp["draft_tokens"].shape
    if "surv" in r:
        r["survival"] = r["surv"]
    else:  # a fixed budget runs no head: those outputs stay untouched (zeros)
        r.update(conf=np.zeros((B, g_)), survival=np.zeros((B, g_)), L0=np.zeros(B, np.int32))
    g = {k: np.array(r[k]) for k in KEYS}
    for k in ("conf", "survival", "p_tok", "q_tok"):
        g[k] = g[k].astype(np.float32)
    g["seq_lens_commit"] = inp["seq_lens"] + r["accept_len"] + 1
    return g


@pytest.mark.parametrize("Tm", [0.0, 1.0])
def test_harness_accepts_the_oracle_and_rejects_changes(Tm):
    inp = W.to_numpy(W.make_inputs(W.TINY, 0, temperature=Tm))
    g = oracle_as_gpu(inp)
    compare_with_oracle(inp, g)
    b = int(np.argmax(g["L"]))
    for key, change in [("out_tokens", lambda x: x.__setitem__((b, 0), (x[b, 0] + 1) % 1024)),
                        ("accept_len", lambda x: x.__setitem__(b, x[b] + 1)),
                        ("L", lambda x: x.__setitem__(b, x[b] - 1)),
                        ("packed_ids", lambda x: x.__setitem__(0, x[0] + 1)),
                        ("seq_lens_commit", lambda x: x.__setitem__(b, x[b] + 1))]:
        bad = {k: v.copy() for k, v in g.items()}
        change(bad[key])
        with pytest.raises(AssertionError):
            compare_with_oracle(inp, bad)
    if Tm > 0:
        bad = {k: v.copy() for k, v in g.items()}
        bad["p_tok"][0] *= 1.01
        with pytest.raises(AssertionError):
            compare_with_oracle(inp, bad)


def test_harness_entropy_variant():
    inp = W.to_numpy(W.make_inputs(W.TINY, 1, temperature=1.0, cost_c=0.02))
    conf, surv, L0, _ = oracle.score_entropy(inp["draft_logits"], 0.3, inp["cost_c"])
    L, _ = oracle.cap(surv, L0, inp["cap_T"])
    cpt = oracle.compact(L, inp["draft_tokens"], inp["last_tokens"], inp["seq_lens"])
    ver = oracle.verify(inp["draft_tokens"], inp["draft_logits"],
                        oracle.ragged_target(inp["target_dense"], L, cpt["row_off"]), L,
                        cpt["row_off"], cpt["draft_off"], inp["temperature"], inp["seed"], EPS_U,
                        inp["seq_lens"])
    g = dict(conf=conf.astype(np.float32), survival=surv.astype(np.float32), L0=L0, L=L, **cpt,
             **{k: ver[k] for k in ("accept_len", "num_emitted", "out_tokens")},
             p_tok=ver["p_tok"].astype(np.float32), q_tok=ver["q_tok"].astype(np.float32),
             seq_lens_commit=ver["seq_lens"])
    compare_with_oracle(inp, g, entropy_theta=0.3)
    bad = dict(g, conf=g["conf"] * np.float32(1.001))
    with pytest.raises(AssertionError):
        compare_with_oracle(inp, bad, entropy_theta=0.3)


@pytest.mark.parametrize("kw", [dict(cap_T=3), dict(cap_T=0), dict(cap_T=-1, fixed_budget=5)])
def test_harness_on_binding_caps_and_fixed_budgets(kw):
    inp = W.to_numpy(W.make_inputs(W.TINY, 2, temperature=1.0, **kw))
    g = oracle_as_gpu(inp)
    if kw.get("fixed_budget", -1) < 0:
        assert g["L"].sum() == min(kw["cap_T"], g["L0"].sum())
    compare_with_oracle(inp, g)
