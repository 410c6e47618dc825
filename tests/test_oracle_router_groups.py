"""Pins for the oracle's group-limited (node-limited) router (CPU only).

The DeepSeek V3/V4 parallel-strategy article (EP section) says V3 limits a
token's 8 experts to the 4 nodes that are best on average, and V4 drops the
limit. The oracle reads a node as a group of consecutive expert ids and "best
on average" as the mean softmax probability of the group's experts. Each test
checks that reading against something other than the oracle's own code:
brute force over all group and expert subsets (arithmetic redone with the
math module), hand-worked examples, and the special cases that reduce to the
plain renormalised top-k."""
import itertools
import math

import numpy as np
import pytest

from oracle import route, ROUTER_RENORM, ROUTER_GROUP_LIMITED


def _probs(row):
    m = max(row)
    ez = [math.exp(v - m) for v in row]
    s = sum(ez)
    return [v / s for v in ez]


def _brute(row, k, G, M):
    """Kept groups: the unique M-subset of groups each of which beats every
    other group (higher mean probability, then lower group id). Chosen
    experts: the unique k-subset of the kept groups' experts each of which
    beats every other kept expert (higher logit, then lower id), in rank
    order. Weights: probabilities of the chosen divided by their sum."""
    E = len(row)
    gs = E // G
    p = _probs(row)
    score = [sum(p[g * gs:(g + 1) * gs]) / gs for g in range(G)]

    def gbeats(a, b):
        return score[a] > score[b] or (score[a] == score[b] and a < b)

    def ebeats(a, b):
        return row[a] > row[b] or (row[a] == row[b] and a < b)

    kept = [S for S in itertools.combinations(range(G), M)
            if all(gbeats(a, b) for a in S for b in range(G) if b not in S)]
    assert len(kept) == 1
    allowed = [e for g in kept[0] for e in range(g * gs, (g + 1) * gs)]
    chosen = [S for S in itertools.combinations(allowed, k)
              if all(ebeats(a, b) for a in S for b in allowed if b not in S)]
    assert len(chosen) == 1
    order = sorted(chosen[0], key=lambda e: (-row[e], e))
    den = sum(p[e] for e in order)
    return order, [p[e] / den for e in order]


@pytest.mark.parametrize("seed", range(4))
def test_group_limited_matches_bruteforce_with_ties(seed):
    # groups of two with small integer logits: exact ties between groups and
    # between experts are frequent (a + b == b + a exactly in IEEE)
    rng = np.random.default_rng(100 + seed)
    for E, G in ((4, 2), (6, 3), (8, 4)):
        for M in range(1, G + 1):
            for k in range(1, min(8, M * (E // G)) + 1):
                L = rng.integers(-2, 3, size=(6, E)).astype(np.float64)
                idx, w = route(L, k, ROUTER_GROUP_LIMITED, n_group=G, topk_group=M)
                for t in range(L.shape[0]):
                    ref_i, ref_w = _brute(list(L[t]), k, G, M)
                    assert list(idx[t]) == ref_i, (E, G, M, k, L[t])
                    np.testing.assert_allclose(w[t], ref_w, rtol=0, atol=1e-14)


def test_group_limited_matches_bruteforce_continuous():
    rng = np.random.default_rng(7)
    for E, G, M, k in ((12, 4, 2, 3), (16, 8, 3, 5), (9, 3, 1, 2), (16, 4, 4, 8)):
        L = 2.0 * rng.standard_normal((25, E))
        idx, w = route(L, k, ROUTER_GROUP_LIMITED, n_group=G, topk_group=M)
        for t in range(25):
            ref_i, ref_w = _brute(list(L[t]), k, G, M)
            assert list(idx[t]) == ref_i
            np.testing.assert_allclose(w[t], ref_w, rtol=0, atol=1e-14)


def test_group_of_the_best_expert_can_lose():
    # group 0 = {2, -6}, group 1 = {1.5, 1.5}: the best single expert (0) sits
    # in the group with the lower average probability, (e^2 + e^-6) / 2 <
    # (2 e^1.5) / 2, so the choice is expert 2 (equal to 3; lower id first)
    L = np.array([[2.0, -6.0, 1.5, 1.5]])
    assert (math.exp(2) + math.exp(-6)) < 2 * math.exp(1.5)
    idx, w = route(L, 1, ROUTER_GROUP_LIMITED, n_group=2, topk_group=1)
    assert idx.tolist() == [[2]] and w.tolist() == [[1.0]]


def test_group_score_is_mean_probability_not_mean_logit():
    # mean logits: group 0 = 0, group 1 = 1; mean probabilities: group 0 wins
    # (e^4 + e^-4 > 2e). The two readings choose different experts.
    L = np.array([[4.0, -4.0, 1.0, 1.0]])
    idx, w = route(L, 2, ROUTER_GROUP_LIMITED, n_group=2, topk_group=1)
    assert idx.tolist() == [[0, 1]]
    den = math.exp(4) + math.exp(-4)
    np.testing.assert_allclose(w[0], [math.exp(4) / den, math.exp(-4) / den], rtol=0, atol=1e-15)


def test_tied_groups_lower_group_id_first():
    L = np.array([[1.0, 0.0, 0.0, 1.0]])     # both groups hold {0, 1}
    idx, _ = route(L, 1, ROUTER_GROUP_LIMITED, n_group=2, topk_group=1)
    assert idx.tolist() == [[0]]


def test_worked_example_three_groups():
    # groups {5, 0}, {3, 3}, {-1, 4.5}: averages e^5+1 > e^-1+e^4.5 > 2e^3,
    # so groups 0 and 2 stay; the top 3 of {5, 0, -1, 4.5} are experts 0, 5, 1
    # although experts 2 and 3 (logit 3) beat expert 1 globally
    L = np.array([[5.0, 0.0, 3.0, 3.0, -1.0, 4.5]])
    idx, w = route(L, 3, ROUTER_GROUP_LIMITED, n_group=3, topk_group=2)
    assert idx.tolist() == [[0, 5, 1]]
    num = [math.exp(5.0), math.exp(4.5), math.exp(0.0)]
    np.testing.assert_allclose(w[0], [v / sum(num) for v in num], rtol=0, atol=1e-15)


def test_one_group_is_plain_renormalised_topk():
    rng = np.random.default_rng(3)
    L = rng.standard_normal((40, 16))
    for k in (1, 2, 8):
        i0, w0 = route(L, k, ROUTER_RENORM, pre_k=8)
        i1, w1 = route(L, k, ROUTER_GROUP_LIMITED, n_group=1, topk_group=1)
        assert np.array_equal(i0, i1)
        np.testing.assert_allclose(w1, w0, rtol=0, atol=1e-15)


def test_all_groups_kept_is_plain_renormalised_topk():
    rng = np.random.default_rng(4)
    L = rng.integers(-3, 4, size=(40, 16)).astype(np.float64)
    for G in (2, 4, 16):
        i0, w0 = route(L, 4, ROUTER_RENORM, pre_k=8)
        i1, w1 = route(L, 4, ROUTER_GROUP_LIMITED, n_group=G, topk_group=G)
        assert np.array_equal(i0, i1)
        np.testing.assert_allclose(w1, w0, rtol=0, atol=1e-15)


def test_singleton_groups_reduce_to_plain_topk():
    # one expert per group: the best M groups are the best M experts, and the
    # top k of those is the plain top k whenever M >= k
    rng = np.random.default_rng(5)
    L = rng.standard_normal((40, 12))
    for M in (3, 5, 12):
        i0, _ = route(L, 3, ROUTER_RENORM, pre_k=8)
        i1, _ = route(L, 3, ROUTER_GROUP_LIMITED, n_group=12, topk_group=M)
        assert np.array_equal(i0, i1)


def test_invariants_on_skewed_logits():
    rng = np.random.default_rng(6)
    E, G, M, k = 64, 8, 3, 8
    L = rng.standard_normal((300, E)) + np.log(1.0 / np.arange(1, E + 1))[rng.permutation(E)]
    idx, w = route(L, k, ROUTER_GROUP_LIMITED, n_group=G, topk_group=M)
    gs = E // G
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    for t in range(300):
        groups = set(int(e) // gs for e in idx[t])
        assert len(groups) <= M
        assert len(set(idx[t].tolist())) == k
        for e in idx[t]:
            for o in range(E):
                if o in idx[t] or o // gs not in groups:
                    continue
                assert L[t, e] >= L[t, o]


def test_group_limited_rejects_bad_shapes():
    L = np.zeros((2, 6))
    with pytest.raises(ValueError):
        route(L, 1, ROUTER_GROUP_LIMITED, n_group=4, topk_group=1)   # 4 does not divide 6
    with pytest.raises(ValueError):
        route(L, 3, ROUTER_GROUP_LIMITED, n_group=3, topk_group=1)   # k > 1 group of 2
    with pytest.raises(ValueError):
        route(L, 1, ROUTER_GROUP_LIMITED, n_group=3, topk_group=4)
