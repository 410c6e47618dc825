"""Pins for the oracle's gate and router (CPU only).

Each test checks the oracle against something other than itself: brute force
over all k-subsets, closed forms written with Python's math module, and
special cases (k = E, pre_k = E, huge logits)."""
import itertools
import math

import numpy as np
import pytest

from oracle import gate_logits, route, ROUTER_RENORM, ROUTER_PREK_SOFTMAX


def _beats(a, b, L):
    """True if expert a ranks before expert b: larger logit, then lower id."""
    return L[a] > L[b] or (L[a] == L[b] and a < b)


def _brute_topk(L, k):
    """The unique k-subset every member of which beats every non-member,
    found by trying all C(E, k) subsets; then ordered by the same rule."""
    E = len(L)
    winners = []
    for S in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in S]
        if all(_beats(a, b, L) for a in S for b in rest):
            winners.append(S)
    assert len(winners) == 1
    S = list(winners[0])
    # insertion sort with the ranking rule
    out = []
    for e in S:
        i = 0
        while i < len(out) and _beats(out[i], e, L):
            i += 1
        out.insert(i, e)
    return out


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_bruteforce_with_ties(seed):
    rng = np.random.default_rng(seed)
    for E in range(1, 9):
        for k in range(1, min(E, 8) + 1):
            # small integers make exact ties common
            L = rng.integers(-3, 4, size=(5, E)).astype(np.float64)
            idx, _ = route(L, k, ROUTER_RENORM, pre_k=8)
            for t in range(L.shape[0]):
                assert list(idx[t]) == _brute_topk(list(L[t]), k)


def test_topk_bruteforce_continuous_values():
    rng = np.random.default_rng(11)
    L = rng.standard_normal((50, 8))
    for k in (1, 2, 3, 8):
        idx, _ = route(L, k, ROUTER_RENORM, pre_k=8)
        for t in range(50):
            assert list(idx[t]) == _brute_topk(list(L[t]), k)


def test_renormalised_weights_sum_to_one():
    rng = np.random.default_rng(1)
    L = rng.standard_normal((200, 64)) * 3
    for k in (1, 2, 8):
        _, w = route(L, k, ROUTER_RENORM)
        assert np.all(np.abs(w.sum(1) - 1.0) <= 1e-12)
        assert np.all(w > 0)
        assert np.all(np.diff(w, axis=1) <= 0)     # slots in descending order


def test_renorm_equals_softmax_over_chosen_logits():
    """Closed form: dividing the chosen full-softmax probabilities by their sum
    equals a softmax taken over the chosen logits alone."""
    rng = np.random.default_rng(2)
    L = rng.standard_normal((40, 16)) * 2
    idx, w = route(L, 3, ROUTER_RENORM)
    for t in range(40):
        z = [L[t, e] for e in idx[t]]
        den = sum(math.exp(v) for v in z)
        for j, v in enumerate(z):
            assert abs(w[t, j] - math.exp(v) / den) <= 1e-14


def test_renorm_independent_of_pre_k():
    """Partial top-8 followed by exact selection gives the same experts and
    weights as selecting from the full sorted list."""
    rng = np.random.default_rng(3)
    L = rng.standard_normal((100, 32))
    a = route(L, 2, ROUTER_RENORM, pre_k=8)
    b = route(L, 2, ROUTER_RENORM, pre_k=32)
    assert np.array_equal(a[0], b[0])
    assert np.allclose(a[1], b[1], rtol=0, atol=1e-15)


def test_k_equals_E_gives_full_softmax():
    rng = np.random.default_rng(4)
    L = rng.standard_normal((10, 6))
    idx, w = route(L, 6, ROUTER_RENORM, pre_k=8)
    for t in range(10):
        den = sum(math.exp(v) for v in L[t])
        for j in range(6):
            assert abs(w[t, j] - math.exp(L[t, idx[t, j]]) / den) <= 1e-14


def test_prek_softmax_weights():
    """Softmax over the 8 largest logits, first k kept without renormalising:
    equals exp(L_j) / sum over the top-8 of exp(L_i)."""
    rng = np.random.default_rng(5)
    L = rng.standard_normal((30, 64)) * 2
    idx, w = route(L, 2, ROUTER_PREK_SOFTMAX, pre_k=8)
    for t in range(30):
        top8 = sorted(range(64), key=lambda e: (-L[t, e], e))[:8]
        assert list(idx[t]) == top8[:2]
        den = sum(math.exp(L[t, e]) for e in top8)
        for j in range(2):
            assert abs(w[t, j] - math.exp(L[t, top8[j]]) / den) <= 1e-14
        assert w[t].sum() < 1.0


def test_prek_softmax_with_all_experts_is_full_softmax():
    rng = np.random.default_rng(6)
    L = rng.standard_normal((20, 8))
    idx, w = route(L, 2, ROUTER_PREK_SOFTMAX, pre_k=8)
    for t in range(20):
        den = sum(math.exp(v) for v in L[t])
        for j in range(2):
            assert abs(w[t, j] - math.exp(L[t, idx[t, j]]) / den) <= 1e-14


def test_huge_logits_do_not_overflow():
    """Max subtraction keeps exp() finite: logits near 1000 would overflow
    e^L in fp64."""
    L = np.array([[1000.0, 999.0, 998.0, 990.0]])
    idx, w = route(L, 2, ROUTER_RENORM)
    assert list(idx[0]) == [0, 1]
    assert np.all(np.isfinite(w))
    assert abs(w[0, 0] - 1.0 / (1.0 + math.exp(-1.0))) <= 1e-15
    idx, w = route(L, 2, ROUTER_PREK_SOFTMAX, pre_k=4)
    den = 1 + math.exp(-1) + math.exp(-2) + math.exp(-10)
    assert abs(w[0, 0] - 1.0 / den) <= 1e-15
    assert abs(w[0, 1] - math.exp(-1) / den) <= 1e-15


def test_gate_matches_triple_loop():
    rng = np.random.default_rng(7)
    T, d, E = 5, 7, 3
    x = rng.standard_normal((T, d))
    Wg = rng.standard_normal((d, E))
    b = rng.standard_normal(E)
    L = gate_logits(x, Wg, b)
    for t in range(T):
        for e in range(E):
            s = b[e]
            for i in range(d):
                s += x[t, i] * Wg[i, e]
            assert abs(L[t, e] - s) <= 1e-12


def test_bias_moves_selection():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((64, 16))
    Wg = rng.standard_normal((16, 8)) * 0.1
    b = np.zeros(8)
    b[5] = 100.0
    idx, _ = route(gate_logits(x, Wg, b), 2, ROUTER_RENORM)
    assert np.all(idx[:, 0] == 5)
    idx0, _ = route(gate_logits(x, Wg, None), 2, ROUTER_RENORM)
    assert not np.all(idx0[:, 0] == 5)
