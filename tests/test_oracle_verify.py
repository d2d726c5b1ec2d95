"""Pins for the oracle's verify (accept / resample / bonus / commit).

Sources: "DFlash to DSpark in SGLang", section "Background" (accepted prefix
plus one bonus token) and section "Serving DeepSeek-V4 with SGLang" (the
target's output distribution is unchanged); "SGLang Integrates DSpark ...",
section "The Old Problem with Speculative Decoding: It Breaks Down at Scale"
(speculative sampling, Chen et al. 2023).

The statistical tests replicate one request over many batch slots; each slot
has its own Philox counter (b, k), so the slots are independent draws.
"""
import json
import os

import numpy as np
import pytest
from scipy import special, stats

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))
ALPHA = 1e-3


def test_greedy_worked_example():
    g = GOLDEN["verify_greedy"]
    tgt = np.array(g["target"], np.float32)
    for case in g["cases"]:
        a, tok, _, _, tie = oracle.verify_request(3, case["drafts"], tgt, None, 0.0,
                                                  np.zeros(4), np.zeros(4), np.zeros(4))
        assert (a, tok) == (case["a"], case["token"]), case
        assert tie == 0


def test_sampling_worked_examples():
    for case in GOLDEN["verify_sampling"]["cases"]:
        Tm = case["Tm"]
        tgt = np.array([np.log(case["p"]), np.log(case["p1"])], np.float64) * Tm
        dft = np.array([np.log(case["q"])], np.float64) * Tm
        a, tok, p, q, _ = oracle.verify_request(1, [case["draft"]], tgt.astype(np.float32),
                                                dft.astype(np.float32), Tm,
                                                np.array(case["u"]), np.array(case["u_blk"]),
                                                np.array(case["u_tok"]))
        assert (a, tok) == (case["a"], case["token"]), case["name"]
        np.testing.assert_allclose(p[0], case["p_tok"], atol=1e-6)
        np.testing.assert_allclose(q[0], case["q_tok"], atol=1e-6)


def _runs(runs):
    return np.concatenate([np.full(n, v, np.float64) for n, v in runs]).astype(np.float32)


def test_two_level_draw_worked_examples():
    for case in GOLDEN["verify_sampling"]["two_block_cases"]["cases"]:
        p1 = _runs(case["p1_runs"])
        row0 = np.zeros_like(p1)
        tgt = np.stack([row0, p1])
        a, tok, _, _, _ = oracle.verify_request(1, [5], tgt, row0[None], 1.0,
                                                np.array([0.5, 0.0]),
                                                np.array([0.0, case["u_blk"]]),
                                                np.array([0.0, case["u_tok"]]))
        assert (a, tok) == (1, case["token"]), case


def _ragged(tgt_rows_per_req, L):
    return np.concatenate(tgt_rows_per_req, axis=0)


@pytest.mark.parametrize("seed", range(4))
def test_greedy_is_longest_argmax_prefix(seed):
    rng = np.random.default_rng(seed)
    B, gamma, V = 12, 5, 40
    tgt_dense = rng.integers(-3, 4, (B, gamma + 1, V)).astype(np.float32)  # many ties
    argm = np.argmax(tgt_dense, axis=-1)                                    # first max
    drafts = argm[:, :gamma].copy().astype(np.int32)
    # break the agreement at a random position in some requests
    for b in range(B):
        if rng.random() < 0.7:
            k = rng.integers(0, gamma)
            drafts[b, k] = (drafts[b, k] + 1 + rng.integers(0, V - 1)) % V
    L = rng.integers(0, gamma + 1, B).astype(np.int32)
    cpt = oracle.compact(L, drafts)
    tgt = oracle.ragged_target(tgt_dense, L, cpt["row_off"])
    out = oracle.verify(drafts, np.zeros((B, gamma, V), np.float32), tgt, L, cpt["row_off"],
                        cpt["draft_off"], 0.0, 0)
    for b in range(B):
        a = 0
        while a < L[b] and drafts[b, a] == argm[b, a]:
            a += 1
        assert out["accept_len"][b] == a
        assert out["num_emitted"][b] == a + 1
        assert list(out["out_tokens"][b, :a]) == list(drafts[b, :a])
        assert out["out_tokens"][b, a] == argm[b, a]
        assert np.all(out["out_tokens"][b, a + 1:] == -1)


def test_greedy_drafts_equal_to_argmax_accept_everything():
    rng = np.random.default_rng(1)
    B, gamma, V = 6, 8, 64
    tgt_dense = rng.standard_normal((B, gamma + 1, V)).astype(np.float32)
    drafts = np.argmax(tgt_dense[:, :gamma], axis=-1).astype(np.int32)
    L = np.array([0, 1, 3, 8, 8, 5], np.int32)
    cpt = oracle.compact(L, drafts)
    tgt = oracle.ragged_target(tgt_dense, L, cpt["row_off"])
    out = oracle.verify(drafts, np.zeros((B, gamma, V), np.float32), tgt, L, cpt["row_off"],
                        cpt["draft_off"], 0.0, 0, seq_lens=np.full(B, 10, np.int32))
    np.testing.assert_array_equal(out["accept_len"], L)
    np.testing.assert_array_equal(out["seq_lens"], 10 + L + 1)


@pytest.mark.parametrize("Tm", [1.0, 0.7])
def test_probabilities_are_library_softmax(Tm):
    rng = np.random.default_rng(2)
    B, gamma, V = 5, 4, 50
    tgt_dense = rng.normal(0, 2, (B, gamma + 1, V)).astype(np.float32)
    dft = (tgt_dense[:, :gamma] + rng.normal(0, 0.5, (B, gamma, V))).astype(np.float32)
    drafts = rng.integers(0, V, (B, gamma)).astype(np.int32)
    L = np.array([4, 0, 2, 3, 1], np.int32)
    cpt = oracle.compact(L, drafts)
    tgt = oracle.ragged_target(tgt_dense, L, cpt["row_off"])
    out = oracle.verify(drafts, dft, tgt, L, cpt["row_off"], cpt["draft_off"], Tm, 11)
    for b in range(B):
        for k in range(L[b]):
            P = special.softmax(tgt_dense[b, k].astype(np.float64) / np.float32(Tm))
            Q = special.softmax(dft[b, k].astype(np.float64) / np.float32(Tm))
            j = cpt["draft_off"][b] + k
            np.testing.assert_allclose(out["p_tok"][j], P[drafts[b, k]], rtol=1e-12)
            np.testing.assert_allclose(out["q_tok"][j], Q[drafts[b, k]], rtol=1e-12)


def test_identical_draft_and_target_accept_everything():
    rng = np.random.default_rng(3)
    B, gamma, V = 40, 6, 30
    tgt_dense = rng.normal(0, 2, (B, gamma + 1, V)).astype(np.float32)
    dft = tgt_dense[:, :gamma].copy()
    drafts = rng.integers(0, V, (B, gamma)).astype(np.int32)
    L = rng.integers(0, gamma + 1, B).astype(np.int32)
    cpt = oracle.compact(L, drafts)
    tgt = oracle.ragged_target(tgt_dense, L, cpt["row_off"])
    out = oracle.verify(drafts, dft, tgt, L, cpt["row_off"], cpt["draft_off"], 1.0, 4)
    np.testing.assert_array_equal(out["accept_len"], L)


def _replicate(p_logits, q_logits, bonus_logits, drafts, n, seed, Tm=1.0):
    """n slots of one L=1 request: row 0 holds (p, q), row 1 the bonus p1."""
    V = p_logits.shape[0]
    L = np.ones(n, np.int32)
    tgt = np.empty((2 * n, V), np.float32)
    tgt[0::2] = p_logits
    tgt[1::2] = bonus_logits
    dft = np.broadcast_to(q_logits, (n, 1, V)).astype(np.float32)
    row_off = (2 * np.arange(n + 1)).astype(np.int32)
    draft_off = np.arange(n + 1).astype(np.int32)
    return oracle.verify(np.asarray(drafts, np.int32).reshape(n, 1), dft, tgt, L, row_off,
                         draft_off, Tm, seed)


@pytest.mark.parametrize("V,seed", [(4, 0), (8, 1), (16, 2)])
def test_accept_frequency_is_min_one_p_over_q(V, seed):
    rng = np.random.default_rng(100 + seed)
    zp = rng.normal(0, 1.5, V).astype(np.float32)
    zq = (zp + rng.normal(0, 1.0, V)).astype(np.float32)
    P, Q = special.softmax(zp.astype(np.float64)), special.softmax(zq.astype(np.float64))
    d = int(np.argmax(Q / P))                     # a draft with r < 1
    r = min(1.0, P[d] / Q[d])
    n = 100_000
    out = _replicate(zp, zq, zp, np.full(n, d), n, seed)
    acc = int(np.sum(out["accept_len"] == 1))
    assert stats.binomtest(acc, n, r).pvalue > ALPHA


@pytest.mark.parametrize("V,seed", [(4, 0), (8, 1), (16, 2)])
def test_resampled_tokens_follow_the_normalised_residual(V, seed):
    rng = np.random.default_rng(200 + seed)
    zp = rng.normal(0, 1.5, V).astype(np.float32)
    zq = (zp + rng.normal(0, 1.5, V)).astype(np.float32)
    P, Q = special.softmax(zp.astype(np.float64)), special.softmax(zq.astype(np.float64))
    d = int(np.argmax(Q / P))
    n = 100_000
    z1 = rng.normal(0, 1.5, V).astype(np.float32)   # a different bonus row
    out = _replicate(zp, zq, z1, np.full(n, d), n, seed)
    rej = out["accept_len"] == 0
    toks = out["out_tokens"][rej, 0]
    resid = np.maximum(0.0, P - Q)
    resid /= resid.sum()
    support = resid > 0
    assert np.all(support[toks])                 # never a token with zero residual
    counts = np.bincount(toks, minlength=V)[support]
    assert stats.chisquare(counts, resid[support] * counts.sum()).pvalue > ALPHA


@pytest.mark.parametrize("V,seed,Tm", [(4, 0, 1.0), (8, 1, 1.0), (16, 2, 0.7)])
def test_first_emitted_token_follows_the_target(V, seed, Tm):
    """Speculative-sampling theorem: with the draft drawn from q, the first
    emitted token (accepted draft or resample) is distributed as p."""
    rng = np.random.default_rng(300 + seed)
    zp = rng.normal(0, 1.5, V).astype(np.float32)
    zq = (zp + rng.normal(0, 1.5, V)).astype(np.float32)
    Tm32 = np.float32(Tm)
    P = special.softmax(zp.astype(np.float64) / Tm32)
    Q = special.softmax(zq.astype(np.float64) / Tm32)
    n = 100_000
    drafts = rng.choice(V, size=n, p=Q / Q.sum())
    out = _replicate(zp, zq, zp, drafts, n, seed, Tm=Tm)
    first = out["out_tokens"][:, 0]
    counts = np.bincount(first, minlength=V)
    assert stats.chisquare(counts, P * n).pvalue > ALPHA


@pytest.mark.parametrize("V,seed", [(4, 3), (16, 4)])
def test_bonus_token_follows_the_target(V, seed):
    rng = np.random.default_rng(400 + seed)
    zp = rng.normal(0, 1.5, V).astype(np.float32)
    z1 = rng.normal(0, 1.5, V).astype(np.float32)
    P1 = special.softmax(z1.astype(np.float64))
    n = 100_000
    # the draft is the argmax of p/q with q == p: ratio 1, always accepted
    out = _replicate(zp, zp, z1, np.zeros(n, np.int32), n, seed)
    assert np.all(out["accept_len"] == 1)
    counts = np.bincount(out["out_tokens"][:, 1], minlength=V)
    assert stats.chisquare(counts, P1 * n).pvalue > ALPHA


def test_commit_and_padding():
    rng = np.random.default_rng(5)
    B, gamma, V = 8, 5, 20
    tgt_dense = rng.normal(0, 1, (B, gamma + 1, V)).astype(np.float32)
    dft = (tgt_dense[:, :gamma] + rng.normal(0, 1, (B, gamma, V))).astype(np.float32)
    drafts = rng.integers(0, V, (B, gamma)).astype(np.int32)
    L = rng.integers(0, gamma + 1, B).astype(np.int32)
    cpt = oracle.compact(L, drafts)
    tgt = oracle.ragged_target(tgt_dense, L, cpt["row_off"])
    sl = rng.integers(10, 100, B).astype(np.int32)
    out = oracle.verify(drafts, dft, tgt, L, cpt["row_off"], cpt["draft_off"], 1.0, 6,
                        seq_lens=sl)
    a = out["accept_len"]
    assert np.all((a >= 0) & (a <= L))
    np.testing.assert_array_equal(out["num_emitted"], a + 1)
    np.testing.assert_array_equal(out["seq_lens"], sl + a + 1)
    for b in range(B):
        row = out["out_tokens"][b]
        assert list(row[:a[b]]) == list(drafts[b, :a[b]])
        assert 0 <= row[a[b]] < V
        assert np.all(row[a[b] + 1:] == -1)


def test_oracle_step_on_the_tiny_workload():
    import torch  # noqa: F401  (the generators draw with torch)
    from confidence_driven_speculative_gb300 import workloads
    for Tm in (0.0, 1.0):
        inp = workloads.to_numpy(workloads.make_inputs(workloads.TINY, 0, temperature=Tm))
        res = oracle.step(inp)
        assert res["L"].sum() <= inp["cap_T"]
        assert np.all(res["accept_len"] <= res["L"])
        assert np.all(np.diff(res["surv"], axis=1) <= 0)


def test_inverse_cdf_uses_strict_crossing():
    """The sampled token is the smallest x with C(x) > u' * Z: a target that
    lands exactly on a cumulative sum moves past it, and u' = 0 never picks a
    token of zero weight."""
    V = 4
    zero = np.zeros(V, np.float32)                   # uniform: C = [.25, .5, .75, 1]
    tgt = np.stack([zero, zero])
    for u3, want in [(0.0, 0), (0.25, 1), (0.5, 2), (0.75, 3), (0.99, 3)]:
        a, tok, _, _, _ = oracle.verify_request(1, [0], tgt, zero[None], 1.0,
                                                np.array([0.0, 0.0]), np.array([0.0, 0.3]),
                                                np.array([0.0, u3]))
        assert (a, tok) == (1, want), u3
    # residual max(0, p - q) = [0, 0.4, 0, 0], u' = 0: the first positive weight
    p = np.array([0.1, 0.5, 0.2, 0.2])
    q = np.array([0.2, 0.1, 0.4, 0.3])
    tgt = np.stack([np.log(p), np.log(p)]).astype(np.float32)
    a, tok, _, _, _ = oracle.verify_request(1, [2], tgt, np.log(q)[None].astype(np.float32), 1.0,
                                            np.array([0.9, 0.0]), np.array([0.0, 0.0]),
                                            np.array([0.0, 0.0]))
    assert (a, tok) == (0, 1)


def test_uniforms_are_wired_to_philox_words():
    """Per slot b the accept test uses word 0 of Philox((b, k, 0, 0), (seed, 0))
    and the in-block draw uses word 2 (one block here, so word 1 plays no
    part): r = 1/2 at every slot, so slot b accepts iff u_b < 1/2; after a
    rejection the residual [0.3, 0, 0.1, 0] (mass 0.4) gives token 0 iff
    u''_b * 0.4 < 0.3."""
    from tests.test_oracle_philox import numpy_block
    seed, n = 77, 300
    p = np.array([0.4, 0.1, 0.3, 0.2])
    q = np.array([0.1, 0.2, 0.2, 0.5])                # p(1)/q(1) = 1/2
    zp = np.log(p).astype(np.float32)
    zq = np.log(q).astype(np.float32)
    out = _replicate(zp, zq, zp, np.ones(n, np.int32), n, seed)
    for b in range(n):
        w0, _, w2 = numpy_block((b, 0, 0, 0), (seed, 0))[:3]
        u = int(w0 >> np.uint64(40)) / 2.0**24
        u2 = int(w2 >> np.uint64(40)) / 2.0**24
        if abs(u - 0.5) < 1e-6:
            continue
        assert out["accept_len"][b] == (1 if u < 0.5 else 0), b
        if u >= 0.5 and abs(u2 * 0.4 - 0.3) > 1e-6:
            assert out["out_tokens"][b, 0] == (0 if u2 * 0.4 < 0.3 else 2), b


def _block_rows(V, spec, rest_mass):
    """Probabilities over V ids: `spec` {id: p}, the rest of the mass spread
    evenly over the other ids (rest_mass may be 0: those ids then get a
    logit far enough below the others that their weight is exactly 0 in
    fp64)."""
    p = np.zeros(V)
    for i, v in spec.items():
        p[i] = v
    others = np.ones(V, bool)
    others[list(spec)] = False
    if rest_mass > 0:
        p[others] = rest_mass / others.sum()
        return np.log(p).astype(np.float32)
    z = np.full(V, -2000.0)
    z[~others] = np.log(p[~others])
    return z.astype(np.float32)


def test_block_uniform_is_wired_to_philox_word_1():
    """Rows of two 4096-id blocks.  Residual path: draft id 1 has
    p/q = 1/2, so slot b rejects iff u_b >= 1/2; the residual's only positive
    ids are 5 (mass 0.30, block 0) and 4103 (mass 0.10, block 1), so after a
    rejection the token is 5 iff u'_b * 0.4 < 0.3, u' being word 1 of
    Philox((b, 0, 0, 0), (seed, 0)).  Bonus path (draft = target, always
    accepted): the bonus row has block masses 0.65 / 0.35, so the bonus token
    lies in block 0 iff u' of position 1 is below 0.65.  Swapping words 1 and
    2 fails both."""
    from tests.test_oracle_philox import numpy_block
    V, seed, n = 8192, 91, 300
    zp = _block_rows(V, {1: 0.1, 5: 0.35, 4103: 0.15}, 0.4)
    zq = _block_rows(V, {1: 0.2, 5: 0.05, 4103: 0.05}, 0.7)
    out = _replicate(zp, zq, zp, np.ones(n, np.int32), n, seed)
    checked = 0
    for b in range(n):
        w = numpy_block((b, 0, 0, 0), (seed, 0))
        u = int(w[0] >> np.uint64(40)) / 2.0**24
        u1 = int(w[1] >> np.uint64(40)) / 2.0**24
        if abs(u - 0.5) < 1e-4:
            continue
        assert out["accept_len"][b] == (1 if u < 0.5 else 0), b
        if u >= 0.5 and abs(u1 - 0.75) > 1e-4:
            assert out["out_tokens"][b, 0] == (5 if u1 < 0.75 else 4103), b
            checked += 1
    assert checked > 100
    z1 = _block_rows(V, {10: 0.6, 4116: 0.3}, 0.1)
    out = _replicate(zp, zp, z1, np.ones(n, np.int32), n, seed)
    assert np.all(out["accept_len"] == 1)
    for b in range(n):
        w = numpy_block((b, 1, 0, 0), (seed, 0))
        u1 = int(w[1] >> np.uint64(40)) / 2.0**24
        if abs(u1 - 0.65) > 1e-4:
            assert (out["out_tokens"][b, 1] < 4096) == (u1 < 0.65), b


def test_bonus_draw_across_three_blocks_follows_the_target():
    """chi-square of L = 0 bonus draws from a row whose mass sits on two ids
    in each of three 4096-id blocks (the other ids weigh exactly 0): both
    levels of the draw -- the block by u', the id inside it by u'' -- must
    reproduce p."""
    V, n, seed = 3 * 4096, 20_000, 17
    spec = {3: 0.10, 1000: 0.15, 4100: 0.20, 8000: 0.05, 8200: 0.25, 12000: 0.25}
    z = _block_rows(V, spec, 0.0)
    L = np.zeros(n, np.int32)
    tgt = np.broadcast_to(z, (n, V)).astype(np.float32)
    row_off = np.arange(n + 1, dtype=np.int32)
    draft_off = np.zeros(n + 1, np.int32)
    out = oracle.verify(np.zeros((n, 1), np.int32), np.zeros((n, 1, V), np.float32), tgt, L,
                        row_off, draft_off, 1.0, seed)
    toks = out["out_tokens"][:, 0]
    ids = np.array(sorted(spec))
    assert np.all(np.isin(toks, ids))
    counts = np.array([np.sum(toks == i) for i in ids])
    P = special.softmax(z.astype(np.float64))[ids]
    assert stats.chisquare(counts, P / P.sum() * n).pvalue > ALPHA


def test_residual_draw_across_two_blocks_follows_the_residual():
    """chi-square of residual draws whose positive part max(0, p - q) sits on
    two ids in each of two blocks (4096 ids and a ragged 8): the resampled
    ids follow norm(max(0, p - q)) across the block boundary."""
    V, n, seed = 4096 + 8, 20_000, 23
    zp = _block_rows(V, {50: 0.05, 3: 0.25, 700: 0.20, 4097: 0.30, 4100: 0.15}, 0.05)
    zq = _block_rows(V, {50: 0.60, 3: 0.05, 700: 0.05, 4097: 0.05, 4100: 0.05}, 0.20)
    out = _replicate(zp, zq, zp, np.full(n, 50, np.int32), n, seed)
    rej = out["accept_len"] == 0
    assert rej.sum() > 0.85 * n
    toks = out["out_tokens"][rej, 0]
    P = special.softmax(zp.astype(np.float64))
    Q = special.softmax(zq.astype(np.float64))
    resid = np.maximum(0.0, P - Q)
    ids = np.nonzero(resid > 0)[0]
    assert set(ids.tolist()) == {3, 700, 4097, 4100}
    assert np.all(np.isin(toks, ids))
    counts = np.array([np.sum(toks == i) for i in ids])
    assert stats.chisquare(counts, resid[ids] / resid[ids].sum() * counts.sum()).pvalue > ALPHA
