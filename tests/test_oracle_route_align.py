"""Pins for the oracle's token routing and alignment.

Routing ("token routing", the English original page, Introduction): per token a
softmax over the E router logits, the k experts with the largest logits (ties
go to the lower expert index), weights = the selected probabilities,
renormalised to sum 1 when asked.  Alignment ("data shuffling", same section):
pairs regrouped by expert into contiguous, padded, stable segments.

Pins: brute-force enumeration of k-subsets, numpy's stable argsort, scipy's
softmax, numpy's bincount and structural invariants.
"""
import itertools

import numpy as np
import pytest
from scipy.special import softmax

import oracle


def brute_topk(row, k):
    """Unique k-subset whose members all precede all non-members under
    (logit desc, index asc); slots ordered the same way."""
    E = len(row)

    def before(a, b):
        return row[a] > row[b] or (row[a] == row[b] and a < b)

    winners = []
    for S in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in S]
        if all(before(a, b) for a in S for b in rest):
            winners.append(S)
    assert len(winners) == 1
    S = list(winners[0])
    # order inside the subset
    S.sort(key=lambda e: (-float(row[e]), e))
    return S


@pytest.mark.parametrize("E", [1, 2, 3, 5, 8])
def test_topk_brute_force_with_ties(E):
    rng = np.random.default_rng(E)
    choices = np.array([-1.0, -0.0, 0.0, 0.5, 0.5, 1.0, 2.0], np.float32)
    for trial in range(60):
        T = 4
        logits = rng.choice(choices, size=(T, E)).astype(np.float32)
        for k in range(1, E + 1):
            ids, _ = oracle.route_topk(logits, k, True)
            for t in range(T):
                assert list(ids[t]) == brute_topk(logits[t], k), (logits[t], k)


def test_topk_matches_stable_argsort():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((300, 64)).astype(np.float32)
    logits[::7, 5] = logits[::7, 9]  # exact duplicates
    logits[::11] = 0.25               # all-equal rows
    for k in (1, 2, 8, 64):
        ids, _ = oracle.route_topk(logits, k, False)
        ref = np.argsort(-logits, axis=1, kind="stable")[:, :k]
        assert np.array_equal(ids, ref)


def test_signed_zero_ties_go_to_lower_index():
    logits = np.array([[-0.0, 0.0, -1.0], [0.0, -0.0, -1.0]], np.float32)
    ids, _ = oracle.route_topk(logits, 1, True)
    assert ids[:, 0].tolist() == [0, 0]


def test_weights_closed_forms():
    rng = np.random.default_rng(4)
    logits = (rng.standard_normal((50, 16)) * 3).astype(np.float32)
    p = softmax(logits.astype(np.float64), axis=1)
    # no renormalisation: weights are the full-softmax probabilities of the picks
    ids, w = oracle.route_topk(logits, 4, False)
    assert np.allclose(w, np.take_along_axis(p, ids, 1), rtol=1e-13, atol=0)
    # renormalised: the same, divided by their sum; sums to 1
    ids2, w2 = oracle.route_topk(logits, 4, True)
    assert np.array_equal(ids, ids2)
    sel = np.take_along_axis(p, ids, 1)
    assert np.allclose(w2, sel / sel.sum(1, keepdims=True), rtol=1e-13, atol=0)
    assert np.allclose(w2.sum(1), 1.0, rtol=0, atol=1e-14)
    # k = E without renormalisation is the dense softmax, in sorted order
    ids3, w3 = oracle.route_topk(logits, 16, False)
    assert np.allclose(w3, np.take_along_axis(p, ids3, 1), rtol=1e-13)
    assert np.allclose(w3.sum(1), 1.0, atol=1e-14)


def test_large_logits_do_not_overflow():
    logits = np.array([[1e30, 1e30, -1e30, 0.0]], np.float32)
    ids, w = oracle.route_topk(logits, 2, True)
    assert ids.tolist() == [[0, 1]]
    assert np.allclose(w, 0.5)


def check_align(ids, E, bm, res):
    T, k = ids.shape
    P = T * k
    flat = ids.ravel()
    counts = np.bincount(flat, minlength=E)
    assert np.array_equal(res["counts"], counts)
    padded = -(-counts // bm) * bm
    assert np.array_equal(res["offsets"], np.concatenate([[0], np.cumsum(padded)]))
    assert res["num_padded"] == padded.sum()
    srt = res["sorted_ids"]
    for e in range(E):
        seg = srt[res["offsets"][e]:res["offsets"][e + 1]]
        real = np.nonzero(flat == e)[0]
        assert np.array_equal(seg[:counts[e]], real)          # stable, ascending
        assert np.all(seg[counts[e]:] == P)                   # sentinel padding
        for b in range(res["offsets"][e] // bm, res["offsets"][e + 1] // bm):
            assert res["tile_expert"][b] == e
    # every pair exactly once
    real = srt[srt < P]
    assert np.array_equal(np.sort(real), np.arange(P))


@pytest.mark.parametrize("E,k,T,bm", [(8, 2, 4, 16), (128, 8, 64, 16), (5, 5, 7, 1),
                                      (3, 1, 100, 4), (256, 8, 32, 64), (1, 1, 9, 8)])
def test_align_invariants(E, k, T, bm):
    rng = np.random.default_rng(E * 31 + k)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    ids, _ = oracle.route_topk(logits, k, True)
    check_align(ids, E, bm, oracle.align(ids, E, bm))


def test_align_skewed_and_empty_experts():
    ids = np.array([[0, 3], [0, 1], [3, 0], [0, 1]], np.int32)
    res = oracle.align(ids, 6, 4)
    check_align(ids, 6, 4, res)
    assert res["counts"].tolist() == [4, 2, 0, 2, 0, 0]
    assert res["sorted_ids"].tolist() == [0, 2, 5, 6, 3, 7, 8, 8, 1, 4, 8, 8]


def test_align_no_tokens():
    ids = np.zeros((0, 2), np.int32)
    res = oracle.align(ids, 4, 16)
    assert res["num_padded"] == 0 and res["counts"].tolist() == [0, 0, 0, 0]
