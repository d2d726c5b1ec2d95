"""Pins for the oracle's batch-wide cap and ragged packing.

Cap: "DFlash to DSpark in SGLang", section "Zero-overhead scheduling and
kernels" (verify-length top-k schedule).  Packing: same page, section "Ragged
verify under full CUDA graphs" (front-packed rows, cu_seqlens offsets).
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def test_cap_worked_example():
    g = GOLDEN["cap"]
    for case in g["cases"]:
        L, _ = oracle.cap(np.array(g["surv"]), np.array(g["L0"]), case["T"])
        assert list(L) == case["L"], case
    t = g["ties"]
    for case in t["cases"]:
        L, _ = oracle.cap(np.array(t["surv"]), np.array(t["L0"]), case["T"])
        assert list(L) == case["L"], case


def _brute_force_best(S, L0, T):
    """Exhaustive search: among all prefix-length vectors L <= L0 with
    sum(L) = min(T, sum(L0)), the one with the largest total survival mass
    sum_b sum_{k<=L_b} S_{b,k} (expected accepted drafts)."""
    B = len(L0)
    target = min(T, int(np.sum(L0)))
    best, best_val = None, -1.0
    for L in itertools.product(*[range(l + 1) for l in L0]):
        if sum(L) != target:
            continue
        val = sum(S[b, :L[b]].sum() for b in range(B))
        if val > best_val + 1e-15:
            best, best_val = L, val
    return np.array(best), best_val


@pytest.mark.parametrize("seed", range(12))
def test_cap_maximises_expected_accepted_drafts(seed):
    rng = np.random.default_rng(seed)
    B, gamma = 3, 4
    conf = rng.uniform(0.3, 1.0, (B, gamma))
    S = np.cumprod(conf, axis=1)
    L0 = rng.integers(0, gamma + 1, B).astype(np.int32)
    for T in range(0, int(L0.sum()) + 2):
        L, _ = oracle.cap(S, L0, T)
        want, want_val = _brute_force_best(S, L0, T)
        got_val = sum(S[b, :L[b]].sum() for b in range(B))
        assert abs(got_val - want_val) < 1e-12
        np.testing.assert_array_equal(L, want)
        assert L.sum() <= T and np.all(L <= L0) and np.all(L >= 0)


def test_cap_negative_means_uncapped_and_zero_means_plain_decode():
    rng = np.random.default_rng(9)
    S = np.cumprod(rng.uniform(0.5, 1, (6, 5)), axis=1)
    L0 = rng.integers(0, 6, 6).astype(np.int32)
    L, _ = oracle.cap(S, L0, -1)
    np.testing.assert_array_equal(L, L0)
    L, _ = oracle.cap(S, L0, 0)
    assert np.all(L == 0)


def test_cap_tie_flag():
    S = np.array([[0.5, 0.1], [0.5 - 1e-7, 0.1]])
    L, tie = oracle.cap(S, np.array([1, 1]), 1, eps=2e-5)
    assert list(L) == [1, 0] and tie == 1
    S = np.array([[0.5, 0.1], [0.4, 0.1]])
    L, tie = oracle.cap(S, np.array([1, 1]), 1, eps=2e-5)
    assert tie == 0


def test_compact_worked_example():
    g = GOLDEN["compact"]
    out = oracle.compact(np.array(g["L"]), np.array(g["draft_tokens"]),
                         np.array(g["last_tokens"]), np.array(g["seq_lens"]))
    for key in ("draft_off", "row_off", "packed_ids", "packed_pos", "row_req", "row_k"):
        assert list(out[key]) == g[key], key


@pytest.mark.parametrize("seed", range(5))
def test_compact_offsets_are_exclusive_scans_and_round_trip(seed):
    rng = np.random.default_rng(seed)
    B, gamma = 17, 6
    L = rng.integers(0, gamma + 1, B).astype(np.int32)
    drafts = rng.integers(0, 1000, (B, gamma)).astype(np.int32)
    last = rng.integers(0, 1000, B).astype(np.int32)
    sl = rng.integers(0, 5000, B).astype(np.int32)
    out = oracle.compact(L, drafts, last, sl)
    np.testing.assert_array_equal(out["draft_off"], np.concatenate([[0], np.cumsum(L)]))
    np.testing.assert_array_equal(out["row_off"], np.concatenate([[0], np.cumsum(L + 1)]))
    np.testing.assert_array_equal(out["row_off"], out["draft_off"] + np.arange(B + 1))
    n = out["row_off"][-1]
    req, kk = out["row_req"][:n], out["row_k"][:n]
    # every (b, j <= L_b) appears exactly once, in request-major order
    assert sorted(zip(req, kk)) == [(b, j) for b in range(B) for j in range(L[b] + 1)]
    assert list(zip(req, kk)) == [(b, j) for b in range(B) for j in range(L[b] + 1)]
    for r in range(n):
        b, j = req[r], kk[r]
        assert out["packed_ids"][r] == (last[b] if j == 0 else drafts[b, j - 1])
        assert out["packed_pos"][r] == sl[b] + j
    assert np.all(out["row_req"][n:] == -1) and np.all(out["packed_ids"][n:] == -1)


def test_compact_without_roots_or_positions():
    out = oracle.compact(np.array([2, 0]), np.array([[5, 6], [7, 8]]))
    assert list(out["packed_ids"][:4]) == [-1, 5, 6, -1]
    assert list(out["packed_pos"][:4]) == [0, 1, 2, 0]


def test_fixed_budget():
    assert list(oracle.fixed_budget(4, 16, 5)) == [5, 5, 5, 5]
    assert list(oracle.fixed_budget(2, 3, 9)) == [3, 3]
    assert list(oracle.fixed_budget(2, 3, 0)) == [0, 0]
