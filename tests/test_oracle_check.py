"""Pins of oracle.check_request: the outcomes a request admits once every
decision within its tolerance window may go either way.

The GPU parity tests use it for requests the oracle flags as near ties: the
GPU's accept length and token must be one of these outcomes, everything else
exact.  Each case below builds rows whose probabilities are known in closed
form (logits log p, temperature 1) and uniforms placed by hand on either side
of a window, so a dropped window, a wrong side or a wrong block fails here.
"""
import numpy as np

import oracle

NEG = -1.0e4  # exp(NEG) is 0 in fp64: a token of zero weight


def rows(*probs, V):
    """fp32 logit rows whose softmax at temperature 1 is the given {id: p}."""
    out = np.full((len(probs), V), NEG, np.float32)
    for i, spec in enumerate(probs):
        for y, p in spec.items():
            out[i, y] = np.log(p)
    return out


def check(L, drafts, tgt, dft, u, u2, u3, a_g, tok_g, Tm=1.0):
    return oracle.check_request(L, np.asarray(drafts, np.int32), tgt, dft, Tm,
                                np.asarray(u, float), np.asarray(u2, float),
                                np.asarray(u3, float), a_g, tok_g)


# One draft, d = 0 with p(d) = 0.25, q(d) = 0.5: r = 0.5.
V4 = 4
TGT = rows({0: 0.25, 1: 0.75}, {2: 1.0}, V=V4)   # row 0 (draft 0), row 1 (bonus)
DFT = rows({0: 0.5, 1: 0.5}, V=V4)


def test_accept_window():
    # u just above r, inside the window: the oracle rejects, accepting is open
    v, kinds = check(1, [0], TGT, DFT, [0.5 + 3e-6, 0.5], [0.5, 0.5], [0.5, 0.5], 1, 2)
    assert v == 0 and kinds[0] == 1
    # outside the window the accept is wrong (an earlier test rejects)
    v, _ = check(1, [0], TGT, DFT, [0.5 + 3e-5, 0.5], [0.5, 0.5], [0.5, 0.5], 1, 2)
    assert v == 2
    # a clear accept (u = 0.1 < r) reported as a rejection at k = 0
    v, _ = check(1, [0], TGT, DFT, [0.1, 0.5], [0.5, 0.5], [0.5, 0.5], 0, 1)
    assert v == 3
    # a_g outside [0, L]
    assert check(1, [0], TGT, DFT, [0.1, 0.5], [0.5, 0.5], [0.5, 0.5], 2, 2)[0] == 1


def test_residual_draw_is_exact_without_a_tie():
    # rejection at k = 0: residual max(0, p - q) = {1: 0.25}: only id 1 is drawn
    assert check(1, [0], TGT, DFT, [0.9, 0.5], [0.3, 0.5], [0.6, 0.5], 0, 1)[0] == 0
    assert check(1, [0], TGT, DFT, [0.9, 0.5], [0.3, 0.5], [0.6, 0.5], 0, 0)[0] == 4
    # every draft accepted: the bonus token of row 1 is id 2
    assert check(1, [0], TGT, DFT, [0.1, 0.5], [0.3, 0.5], [0.6, 0.5], 1, 2)[0] == 0
    assert check(1, [0], TGT, DFT, [0.1, 0.5], [0.3, 0.5], [0.6, 0.5], 1, 1)[0] == 4
    # a token of -1 checks the accept length alone
    assert check(1, [0], TGT, DFT, [0.9, 0.5], [0.3, 0.5], [0.6, 0.5], 0, -1)[0] == 0
    assert check(1, [0], TGT, DFT, [0.9, 0.5], [0.3, 0.5], [0.6, 0.5], 1, -1)[0] == 2


V2B = 2 * 4096  # two sampling blocks
BONUS_2B = rows({7: 0.5, 4100: 0.5}, V=V2B)


def test_block_level_window():
    # t = (0.5 + 1e-7) Z sits 1e-7 Z past the block boundary: block 1 is the
    # crossing, block 0 is within eps_blk Z = 1e-6 Z of it
    v, kinds = check(0, [], BONUS_2B, None, [0.5], [0.5 + 1e-7], [0.5], 0, 4100)
    assert v == 0 and kinds[2] >= 1
    assert check(0, [], BONUS_2B, None, [0.5], [0.5 + 1e-7], [0.5], 0, 7)[0] == 0
    assert check(0, [], BONUS_2B, None, [0.5], [0.5 + 1e-7], [0.5], 0, 5)[0] == 4  # zero weight
    # far from the boundary only block 0's token is drawn
    assert check(0, [], BONUS_2B, None, [0.5], [0.3], [0.5], 0, 7)[0] == 0
    assert check(0, [], BONUS_2B, None, [0.5], [0.3], [0.5], 0, 4100)[0] == 4


BONUS_IN = rows({3: 0.25, 9: 0.25, 5000: 0.5}, V=V2B)


def test_in_block_window():
    # block 0 (mass 0.5); in-block target (0.5 + 1e-7) * 0.5 is 5e-8 past
    # id 3's interval, inside eps_tok * 0.5 = 1e-6
    assert check(0, [], BONUS_IN, None, [0.5], [0.2], [0.5 + 1e-7], 0, 9)[0] == 0
    assert check(0, [], BONUS_IN, None, [0.5], [0.2], [0.5 + 1e-7], 0, 3)[0] == 0
    assert check(0, [], BONUS_IN, None, [0.5], [0.2], [0.5 + 1e-7], 0, 5000)[0] == 4
    # far inside id 9's interval only id 9
    assert check(0, [], BONUS_IN, None, [0.5], [0.2], [0.7], 0, 9)[0] == 0
    assert check(0, [], BONUS_IN, None, [0.5], [0.2], [0.7], 0, 3)[0] == 4


def test_small_residual_mass_opens_the_fallback():
    # p = (0.5 - 2e-6, 0.5 + 2e-6), q = (0.5, 0.5): residual Z = 2e-6 < eps
    tgt = rows({0: 0.5 - 2e-6, 1: 0.5 + 2e-6}, {0: 1.0}, V=V4)
    dft = rows({0: 0.5, 1: 0.5}, V=V4)
    u = [0.999999, 0.5]  # r = 0.999996: rejected (and within the window)
    v, kinds = check(1, [0], tgt, dft, u, [0.5, 0.5], [0.2, 0.5], 0, 1)
    assert v == 0 and kinds[1] == 1
    # id 0 has no residual weight, but the fallback draw from p lands on it
    assert check(1, [0], tgt, dft, u, [0.5, 0.5], [0.2, 0.5], 0, 0)[0] == 0
    # with a large residual mass the fallback is closed
    tgt2 = rows({0: 0.2, 1: 0.8}, {0: 1.0}, V=V4)
    assert check(1, [0], tgt2, dft, [0.9, 0.5], [0.5, 0.5], [0.2, 0.5], 0, 0)[0] == 4
    assert check(1, [0], tgt2, dft, [0.9, 0.5], [0.5, 0.5], [0.2, 0.5], 0, 1)[0] == 0


def test_greedy_is_exact():
    tgt = rows({1: 0.6, 2: 0.4}, {3: 0.9, 0: 0.1}, V=V4)
    # draft 1 is the argmax of row 0: accepted; the bonus is row 1's argmax 3
    assert check(1, [1], tgt, None, [0, 0], [0, 0], [0, 0], 1, 3, Tm=0.0)[0] == 0
    assert check(1, [1], tgt, None, [0, 0], [0, 0], [0, 0], 0, 1, Tm=0.0)[0] == 5
    assert check(1, [1], tgt, None, [0, 0], [0, 0], [0, 0], 1, 0, Tm=0.0)[0] == 5
    # draft 2 is not: rejected at 0, the correction is row 0's argmax 1
    assert check(1, [2], tgt, None, [0, 0], [0, 0], [0, 0], 0, 1, Tm=0.0)[0] == 0


def test_own_outcome_is_always_admitted():
    """On random requests the oracle's own outcome passes its own check, and
    a different token at an untied draw does not."""
    rng = np.random.default_rng(3)
    V, L = 9000, 5
    for trial in range(6):
        tgt = rng.normal(0, 2, (L + 1, V)).astype(np.float32)
        dft = (tgt[:L] + rng.normal(0, 0.5, (L, V))).astype(np.float32)
        drafts = rng.integers(0, V, L).astype(np.int32)
        u, u2, u3 = rng.random(L + 1), rng.random(L + 1), rng.random(L + 1)
        a, tok, _, _, tie = oracle.verify_request(L, drafts, tgt, dft, 1.0, u, u2, u3)
        v, kinds = check(L, drafts, tgt, dft, u, u2, u3, a, tok)
        assert v == 0
        if tie == 0:
            assert check(L, drafts, tgt, dft, u, u2, u3, a, (tok + 1) % V)[0] == 4
            if a < L:
                assert check(L, drafts, tgt, dft, u, u2, u3, a + 1, tok)[0] == 2
            if a > 0:
                assert check(L, drafts, tgt, dft, u, u2, u3, a - 1, tok)[0] == 3
