"""Pins for the oracle's cap-accept audit arm.

Source: "DFlash to DSpark in SGLang", section "The confidence scheduler and
verify modes": cap-accept verifies the whole block like static, commits only
the scheduled window, so its output is compact's, and it records what the
trim gave up; section "Scheduling results": utilization against the ceiling.

The pins tie the arm to those statements and to the speculative-sampling
rule, not to the oracle's own arithmetic: the committed prefix is the
accepted prefix cut at the window, a window at least the block gives the
static result, a greedy commit cut inside the accepted run ends with the
next draft itself, and a sampled commit cut inside the accepted run draws
its last token from the target row at the window, not from the residual.
"""
import numpy as np
import pytest
from scipy import special, stats

import oracle

ALPHA = 1e-3


def _case(seed, B=12, gamma=6, V=24, noise=0.6):
    rng = np.random.default_rng(seed)
    tgt = rng.normal(0, 1.5, (B, gamma + 1, V)).astype(np.float32)
    dft = (tgt[:, :gamma] + rng.normal(0, noise, (B, gamma, V))).astype(np.float32)
    drafts = np.empty((B, gamma), np.int32)
    for b in range(B):
        for k in range(gamma):
            q = special.softmax(dft[b, k].astype(np.float64))
            drafts[b, k] = rng.choice(V, p=q / q.sum())
    return rng, tgt, dft, drafts


def test_greedy_worked_example():
    # V = 8, gamma = 4.  Row k's argmax is set by hand: rows 0..2 agree with
    # drafts d_1..d_3, row 3 does not (argmax 2, draft 6), row 4 is the bonus.
    V, gamma = 8, 4
    drafts = np.array([[3, 5, 1, 6]], np.int32)
    argmax = [3, 5, 1, 2, 7]
    tgt = np.zeros((1, gamma + 1, V), np.float32)
    for k, y in enumerate(argmax):
        tgt[0, k, y] = 4.0
    L = np.array([gamma], np.int32)
    expect = {  # window -> (committed a, emitted tokens)
        0: (0, [3, -1, -1, -1, -1]),
        1: (1, [3, 5, -1, -1, -1]),
        2: (2, [3, 5, 1, -1, -1]),
        3: (3, [3, 5, 1, 2, -1]),
        4: (3, [3, 5, 1, 2, -1]),
        9: (3, [3, 5, 1, 2, -1]),
    }
    for W, (acc, toks) in expect.items():
        out = oracle.verify_cap_accept(drafts, None, tgt, L, [W], 0.0, 0)
        assert out["accept_full"][0] == 3, W
        assert out["accept_len"][0] == acc, W
        assert out["num_emitted"][0] == acc + 1, W
        assert out["out_tokens"][0].tolist() == toks, W
        assert out["audit_totals"].tolist() == [3, acc], W


@pytest.mark.parametrize("Tm", [0.0, 1.0, 0.6])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_commit_is_the_accepted_prefix_cut_at_the_window(Tm, seed):
    rng, tgt, dft, drafts = _case(seed)
    B, gamma = drafts.shape
    if Tm == 0.0:
        # greedy: make some drafts the target's argmax so runs of accepts occur
        for b in range(B):
            run = rng.integers(0, gamma + 1)
            drafts[b, :run] = np.argmax(tgt[b, :run], axis=-1)
    L = np.full(B, gamma, np.int32)
    L[:3] = rng.integers(0, gamma, 3)
    W = rng.integers(-1, gamma + 2, B).astype(np.int32)
    sl = rng.integers(0, 100, B).astype(np.int32)
    out = oracle.verify_cap_accept(drafts, dft, tgt, L, W, Tm, 11 + seed, seq_lens=sl)
    Wc = np.clip(W, 0, L)
    np.testing.assert_array_equal(out["W"], Wc)
    a_full, acc = out["accept_full"], out["accept_len"]
    assert np.all((0 <= a_full) & (a_full <= L))
    np.testing.assert_array_equal(acc, np.minimum(a_full, Wc))
    np.testing.assert_array_equal(out["num_emitted"], acc + 1)
    np.testing.assert_array_equal(out["seq_lens"], sl + acc + 1)
    for b in range(B):
        row = out["out_tokens"][b]
        assert row[:acc[b]].tolist() == drafts[b, :acc[b]].tolist()
        assert 0 <= row[acc[b]] < tgt.shape[-1]
        assert np.all(row[acc[b] + 1:] == -1)
        if Tm == 0.0 and Wc[b] < a_full[b]:
            # cut inside the accepted run: the greedy token at the window is
            # the target's argmax there, which is the next draft itself
            assert row[Wc[b]] == drafts[b, Wc[b]]
    assert out["audit_totals"].tolist() == [int(a_full.sum()), int(acc.sum())]
    assert out["audit_totals"][1] <= out["audit_totals"][0]
    # p_tok / q_tok cover every draft of the full block
    assert out["p_tok"].shape == (int(L.sum()),)


@pytest.mark.parametrize("Tm", [0.0, 0.8])
def test_window_covering_the_block_is_static(Tm):
    _, tgt, dft, drafts = _case(7)
    B, gamma = drafts.shape
    L = np.full(B, gamma, np.int32)
    out = oracle.verify_cap_accept(drafts, dft, tgt, L, L + 3, Tm, 5)
    lay = oracle.compact(L, drafts)
    st = oracle.verify(drafts, dft, oracle.ragged_target(tgt, L, lay["row_off"]), L,
                       lay["row_off"], lay["draft_off"], Tm, 5)
    np.testing.assert_array_equal(out["accept_full"], st["accept_len"])
    np.testing.assert_array_equal(out["accept_len"], st["accept_len"])
    np.testing.assert_array_equal(out["out_tokens"], st["out_tokens"])
    np.testing.assert_array_equal(out["p_tok"], st["p_tok"])


@pytest.mark.parametrize("V,seed", [(6, 0), (12, 1)])
def test_token_at_a_window_inside_the_accepted_run_follows_the_target(V, seed):
    """Slots whose first draft is accepted, committed with window 1: the full
    verify may accept or reject draft 2, but the emitted token is drawn from
    the target row at the window (compact's bonus), never from the
    residual of that row."""
    rng = np.random.default_rng(500 + seed)
    n, gamma = 60_000, 2
    z0 = rng.normal(0, 1.0, V).astype(np.float32)
    z1 = rng.normal(0, 1.5, V).astype(np.float32)
    zq1 = (z1 + rng.normal(0, 2.0, V)).astype(np.float32)
    P1 = special.softmax(z1.astype(np.float64))
    Q1 = special.softmax(zq1.astype(np.float64))
    tgt = np.empty((n, gamma + 1, V), np.float32)
    tgt[:, 0], tgt[:, 1], tgt[:, 2] = z0, z1, z0
    dft = np.empty((n, gamma, V), np.float32)
    dft[:, 0], dft[:, 1] = z0, zq1          # q == p on row 0: draft 1 always accepted
    drafts = np.empty((n, gamma), np.int32)
    drafts[:, 0] = 0
    drafts[:, 1] = int(np.argmax(Q1 / P1))  # r < 1 on row 1: rejected now and then
    L = np.full(n, gamma, np.int32)
    out = oracle.verify_cap_accept(drafts, dft, tgt, L, np.ones(n, np.int32), 1.0, 17 + seed)
    assert np.all(out["accept_len"] == 1)
    rejected = out["accept_full"] == 1
    assert 0 < rejected.sum() < n             # both outcomes of the full verify occur
    counts = np.bincount(out["out_tokens"][:, 1], minlength=V)
    assert stats.chisquare(counts, P1 * n).pvalue > ALPHA
