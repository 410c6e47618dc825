"""Pins for the oracle's soft-gating router (CPU only).

The Deepseek-MoE sync-tax article (section 3.3) replaces hard top-k with soft
gating: the gate's logits are turned into a probability vector by
Gumbel-Softmax sampling and every expert output is weighted by it (none is
dropped). The oracle's reading: w = softmax((L + g) / tau) over all E, g the
Gumbel samples passed in, slot j = expert j. The pins: closed forms written
with the math module, the temperature limits, invariances, the whole layer
against a direct dense sum over experts, and the Gumbel-max property of the
generator's draws."""
import math

import numpy as np
import pytest

import oracle
from oracle import route, ROUTER_RENORM, ROUTER_SOFT_GUMBEL


def test_zero_noise_unit_temperature_is_the_full_softmax():
    rng = np.random.default_rng(1)
    L = rng.standard_normal((30, 8)) * 3
    idx, w = route(L, 8, ROUTER_SOFT_GUMBEL, gumbel=np.zeros_like(L), tau=1.0)
    assert np.array_equal(idx, np.broadcast_to(np.arange(8), (30, 8)))
    for t in range(30):
        m = max(L[t])
        ez = [math.exp(v - m) for v in L[t]]
        np.testing.assert_allclose(w[t], [v / sum(ez) for v in ez], rtol=0, atol=1e-15)
    # and the renormalised router with k = E gives the same numbers, in rank order
    ir, wr = route(L, 8, ROUTER_RENORM, pre_k=8)
    back = np.take_along_axis(w, ir.astype(np.int64), axis=1)
    np.testing.assert_allclose(back, wr, rtol=0, atol=1e-15)


def test_two_experts_closed_form():
    rng = np.random.default_rng(2)
    L = rng.standard_normal((40, 2))
    g = rng.gumbel(size=(40, 2))
    for tau in (0.3, 1.0, 2.5):
        _, w = route(L, 2, ROUTER_SOFT_GUMBEL, gumbel=g, tau=tau)
        tf = float(np.float32(tau))
        for t in range(40):
            a = (L[t, 0] + g[t, 0]) / tf
            b = (L[t, 1] + g[t, 1]) / tf
            assert abs(w[t, 0] - 1.0 / (1.0 + math.exp(b - a))) < 1e-15
            assert abs(w[t, 0] + w[t, 1] - 1.0) < 1e-15


def test_low_temperature_is_one_hot_at_the_gumbel_max():
    rng = np.random.default_rng(3)
    L = rng.standard_normal((50, 16))
    g = rng.gumbel(size=(50, 16))
    _, w = route(L, 16, ROUTER_SOFT_GUMBEL, gumbel=g, tau=1e-4)
    hot = np.argmax(L + g, axis=1)
    np.testing.assert_allclose(w, np.eye(16)[hot], rtol=0, atol=1e-12)


def test_high_temperature_is_uniform():
    rng = np.random.default_rng(4)
    L = rng.standard_normal((10, 16))
    _, w = route(L, 16, ROUTER_SOFT_GUMBEL, gumbel=rng.gumbel(size=(10, 16)), tau=1e9)
    np.testing.assert_allclose(w, 1.0 / 16, rtol=0, atol=1e-9)


def test_shift_and_scale_invariance():
    rng = np.random.default_rng(5)
    L = rng.standard_normal((20, 8))
    g = rng.gumbel(size=(20, 8))
    _, w = route(L, 8, ROUTER_SOFT_GUMBEL, gumbel=g, tau=0.5)
    _, w2 = route(L + 7.25, 8, ROUTER_SOFT_GUMBEL, gumbel=g - 3.5, tau=0.5)
    np.testing.assert_allclose(w2, w, rtol=0, atol=1e-14)
    _, w3 = route(4 * L, 8, ROUTER_SOFT_GUMBEL, gumbel=4 * g, tau=2.0)
    np.testing.assert_allclose(w3, w, rtol=0, atol=1e-14)
    assert np.all(w > 0) and np.all(np.abs(w.sum(1) - 1) < 1e-12)


def test_forward_is_the_dense_weighted_sum_over_all_experts():
    from workloads import MoEConfig, make_inputs
    cfg = MoEConfig("soft", T=12, d=64, E=4, k=4, f=64, dtype="f32", router=ROUTER_SOFT_GUMBEL,
                    tau=0.7, seed=8)
    inp = make_inputs(cfg)
    res = oracle.forward(cfg, inp)
    x = inp["x"].double().numpy()
    L = x @ inp["Wg"].double().numpy() + inp["bias"].double().numpy()
    z = (L + inp["gumbel"].double().numpy()) / float(np.float32(0.7))
    p = np.exp(z - z.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    ref = np.zeros((12, 64))
    for e in range(4):
        h = x @ inp["W1"][e].double().numpy()
        h = h / (1 + np.exp(-h))
        h = h.astype(np.float32).astype(np.float64)      # H stored in fp32
        ref += p[:, e:e + 1] * (h @ inp["W2"][e].double().numpy())
    np.testing.assert_allclose(res["out"], ref, rtol=0, atol=1e-12)
    # every expert receives every token, in token order
    assert res["counts"].tolist() == [12] * 4
    assert np.array_equal(res["src"], np.tile(np.arange(12), 4))
    tok = oracle.forward_tokens(cfg, inp, np.array([3, 11]))
    np.testing.assert_allclose(tok["out"], res["out"][[3, 11]], rtol=0, atol=1e-12)


def test_generator_draws_are_gumbel():
    # Gumbel-max: argmax(L + g) is distributed as softmax(L) when g is
    # standard Gumbel. 40000 draws of 4 experts: each frequency within 4
    # standard errors.
    from workloads import MoEConfig, make_inputs
    cfg = MoEConfig("g", T=40000, d=64, E=4, k=4, f=64, dtype="f32", router=ROUTER_SOFT_GUMBEL,
                    seed=9)
    g = make_inputs(cfg)["gumbel"].double().numpy()
    L = np.array([0.5, -0.25, 1.0, 0.0])
    p = np.exp(L) / np.exp(L).sum()
    freq = np.bincount(np.argmax(L + g, axis=1), minlength=4) / g.shape[0]
    se = np.sqrt(p * (1 - p) / g.shape[0])
    assert np.all(np.abs(freq - p) < 4 * se), (freq, p)
    # the mean of a standard Gumbel is the Euler-Mascheroni constant
    assert abs(g.mean() - 0.5772156649) < 4 * (math.pi / math.sqrt(6)) / math.sqrt(g.size)


def test_soft_router_rejects_bad_arguments():
    L = np.zeros((3, 4))
    with pytest.raises(ValueError):
        route(L, 2, ROUTER_SOFT_GUMBEL, gumbel=np.zeros((3, 4)))       # k != E
    with pytest.raises(ValueError):
        route(L, 4, ROUTER_SOFT_GUMBEL, gumbel=None)
    with pytest.raises(ValueError):
        route(L, 4, ROUTER_SOFT_GUMBEL, gumbel=np.zeros((3, 4)), tau=0.0)


def test_huge_logits_stay_finite():
    L = np.array([[1000.0, 999.0, 0.0, -1000.0]])
    _, w = route(L, 4, ROUTER_SOFT_GUMBEL, gumbel=np.zeros_like(L), tau=1.0)
    e = math.exp(-1.0)
    np.testing.assert_allclose(w[0], [1 / (1 + e), e / (1 + e), 0.0, 0.0], rtol=0, atol=1e-15)
