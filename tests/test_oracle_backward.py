"""Pins for the oracle's backward pass (CPU only).

The gradients of the scalar <out, dout> are checked against central finite
differences of a forward composed from the oracle's own steps with no storage
rounding (a rounding would make the difference quotient meaningless), on tiny
layers for every router mode, with perturbations too small to change any
expert choice (entries whose perturbation would change the routing are
skipped). The router Jacobians are checked the same way on the weights alone;
SiLU's derivative against its difference quotient; and special cases: the
gradient is linear in dout, a single expert has no router gradient, an
expert with no rows gets zero weight gradients."""
import numpy as np
import pytest

import oracle
from oracle import (ROUTER_GROUP_LIMITED, ROUTER_PREK_SOFTMAX, ROUTER_RENORM,
                    ROUTER_SOFT_GUMBEL)
from workloads import MoEConfig

EPS = 1e-6


def _cfg(router=ROUTER_RENORM, T=6, d=8, E=4, k=2, f=6, pre_k=3, **kw):
    return MoEConfig(f"bwd_pin_{router}", T=T, d=d, E=E, k=k, f=f, dtype="f32", router=router,
                     pre_k=pre_k, **kw)


def _inputs(cfg, seed):
    rng = np.random.default_rng(seed)
    a = {"x": rng.standard_normal((cfg.T, cfg.d)),
         "Wg": rng.standard_normal((cfg.d, cfg.E)) / np.sqrt(cfg.d) * 3.0,
         "bias": rng.standard_normal(cfg.E) * 0.5,
         "W1": rng.standard_normal((cfg.E, cfg.d, cfg.f)) / np.sqrt(cfg.d),
         "W2": rng.standard_normal((cfg.E, cfg.f, cfg.d)) / np.sqrt(cfg.f)}
    if cfg.router == ROUTER_SOFT_GUMBEL:
        a["gumbel"] = rng.gumbel(size=(cfg.T, cfg.E))
    return a


def _exact_forward(cfg, a):
    """The layer from the oracle's steps, H unrounded."""
    L = oracle.gate_logits(a["x"], a["Wg"], a["bias"])
    idx, w = oracle.route(L, cfg.k, cfg.router, cfg.pre_k, getattr(cfg, "n_group", 1),
                          getattr(cfg, "topk_group", 1), a.get("gumbel"),
                          getattr(cfg, "tau", 1.0))
    counts, offsets, pos, src = oracle.dispatch(idx, cfg.E)
    Y = np.zeros((idx.size, cfg.d))
    for e in range(cfg.E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            Y[lo:hi], _ = oracle.expert_ffn_rows(a["x"][src[lo:hi]], a["W1"][e], a["W2"][e],
                                                 "exact")
    out = oracle.combine(Y, pos, w)
    return {"L": L, "topk_idx": idx, "topk_w": w, "counts": counts, "offsets": offsets,
            "pos": pos, "src": src, "Y": Y, "out": out}


def _check_fd(cfg, seed, n_samples=12):
    a = _inputs(cfg, seed)
    rng = np.random.default_rng(seed + 100)
    dout = rng.standard_normal((cfg.T, cfg.d))
    fwd = _exact_forward(cfg, a)
    grads = oracle.backward(cfg, a, fwd, dout, h_storage="exact")
    names = {"x": "dx", "Wg": "dWg", "bias": "dbias", "W1": "dW1", "W2": "dW2"}
    checked = 0
    for name, gname in names.items():
        arr = a[name]
        flat = arr.reshape(-1)
        for i in rng.choice(flat.size, size=min(n_samples, flat.size), replace=False):
            old = flat[i]
            flat[i] = old + EPS
            fp = _exact_forward(cfg, a)
            flat[i] = old - EPS
            fm = _exact_forward(cfg, a)
            flat[i] = old
            if not (np.array_equal(fp["topk_idx"], fwd["topk_idx"]) and
                    np.array_equal(fm["topk_idx"], fwd["topk_idx"])):
                continue              # the perturbation changes a choice
            num = ((fp["out"] - fm["out"]) * dout).sum() / (2 * EPS)
            ana = grads[gname].reshape(-1)[i]
            assert abs(num - ana) <= 1e-6 * max(1.0, abs(num)), (name, i, num, ana)
            checked += 1
    assert checked >= 3 * n_samples


@pytest.mark.parametrize("seed", [0, 1])
def test_finite_differences_renorm(seed):
    _check_fd(_cfg(ROUTER_RENORM), seed)


@pytest.mark.parametrize("seed", [2, 3])
def test_finite_differences_top_prek_softmax(seed):
    _check_fd(_cfg(ROUTER_PREK_SOFTMAX, E=6, k=2, pre_k=4), seed)


def test_finite_differences_group_limited():
    _check_fd(_cfg(ROUTER_GROUP_LIMITED, E=8, k=2, n_group=4, topk_group=2), 4)


def test_finite_differences_soft_gating():
    _check_fd(_cfg(ROUTER_SOFT_GUMBEL, E=4, k=4, tau=0.7), 5)


def test_finite_differences_k_equals_one_and_uneven_experts():
    _check_fd(_cfg(ROUTER_RENORM, T=9, E=5, k=1, pre_k=1), 6)


@pytest.mark.parametrize("router,k,pre_k", [(ROUTER_RENORM, 3, 3), (ROUTER_PREK_SOFTMAX, 2, 5),
                                            (ROUTER_SOFT_GUMBEL, 6, 6)])
def test_router_jacobian(router, k, pre_k):
    rng = np.random.default_rng(7)
    T, E = 5, 6
    L = rng.standard_normal((T, E)) * 2
    g = rng.gumbel(size=(T, E)) if router == ROUTER_SOFT_GUMBEL else None
    tau = 0.8
    idx, w = oracle.route(L, k, router, pre_k, gumbel=g, tau=tau)
    dw = rng.standard_normal(w.shape)
    dL = oracle.router_backward(L, idx, w, dw, router, pre_k, tau)
    for t in range(T):
        for e in range(E):
            Lp, Lm = L.copy(), L.copy()
            Lp[t, e] += EPS
            Lm[t, e] -= EPS
            ip, wp = oracle.route(Lp, k, router, pre_k, gumbel=g, tau=tau)
            im, wm = oracle.route(Lm, k, router, pre_k, gumbel=g, tau=tau)
            assert np.array_equal(ip, idx) and np.array_equal(im, idx)
            num = ((wp - wm) * dw).sum() / (2 * EPS)
            assert abs(num - dL[t, e]) <= 1e-7, (t, e, num, dL[t, e])


def test_silu_grad_is_the_derivative():
    z = np.linspace(-30, 30, 601)
    num = (oracle.moe_oracle.silu(z + EPS) - oracle.moe_oracle.silu(z - EPS)) / (2 * EPS)
    np.testing.assert_allclose(oracle.silu_grad(z), num, rtol=0, atol=1e-8)
    assert oracle.silu_grad(np.array([0.0]))[0] == 0.5


def test_linear_in_dout():
    cfg = _cfg(ROUTER_RENORM)
    a = _inputs(cfg, 8)
    fwd = _exact_forward(cfg, a)
    rng = np.random.default_rng(9)
    g1, g2 = rng.standard_normal((2, cfg.T, cfg.d))
    b1 = oracle.backward(cfg, a, fwd, g1, h_storage="exact")
    b2 = oracle.backward(cfg, a, fwd, g2, h_storage="exact")
    b12 = oracle.backward(cfg, a, fwd, 2 * g1 - 3 * g2, h_storage="exact")
    for n in ("dx", "dWg", "dbias", "dW1", "dW2"):
        np.testing.assert_allclose(b12[n], 2 * b1[n] - 3 * b2[n], rtol=1e-12, atol=1e-12)


def test_single_expert_has_no_router_gradient():
    cfg = _cfg(ROUTER_RENORM, E=1, k=1, pre_k=1)
    a = _inputs(cfg, 10)
    fwd = _exact_forward(cfg, a)
    g = oracle.backward(cfg, a, fwd, np.ones((cfg.T, cfg.d)), h_storage="exact")
    assert np.all(g["dL"] == 0) and np.all(g["dWg"] == 0) and np.all(g["dbias"] == 0)
    # with one expert and weight 1 the layer is a dense FFN: dW2 = H^T dout
    z = a["x"] @ a["W1"][0]
    np.testing.assert_allclose(g["dW2"][0], oracle.moe_oracle.silu(z).T @ np.ones((cfg.T, cfg.d)),
                               rtol=1e-12)


def test_expert_without_rows_gets_zero_gradients():
    cfg = _cfg(ROUTER_RENORM, E=4, k=1, pre_k=1)
    a = _inputs(cfg, 11)
    a["bias"] = np.array([0.0, 0.0, 0.0, -1e3])       # expert 3 is never chosen
    fwd = _exact_forward(cfg, a)
    assert fwd["counts"][3] == 0
    g = oracle.backward(cfg, a, fwd, np.ones((cfg.T, cfg.d)), h_storage="exact")
    assert np.all(g["dW1"][3] == 0) and np.all(g["dW2"][3] == 0) and g["dbias"][3] == 0


def test_fp8_payloads_have_no_backward():
    cfg = _cfg(ROUTER_RENORM, payload_fp8=1)
    with pytest.raises(ValueError):
        oracle.backward(cfg, _inputs(cfg, 0), {}, np.zeros((cfg.T, cfg.d)))


@pytest.mark.parametrize("router", [ROUTER_RENORM, ROUTER_PREK_SOFTMAX, ROUTER_SOFT_GUMBEL])
def test_token_subset_equals_the_whole_layer(router):
    cfg = _cfg(router, T=10, E=6, k=6 if router == ROUTER_SOFT_GUMBEL else 2, pre_k=4)
    a = _inputs(cfg, 12)
    dout = np.random.default_rng(13).standard_normal((cfg.T, cfg.d))
    full = oracle.backward(cfg, a, oracle.forward(cfg, a), dout)
    sub = oracle.backward_tokens(cfg, a, dout, [7, 2, 5])
    np.testing.assert_allclose(sub["dx"], full["dx"][[7, 2, 5]], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sub["dL"], full["dL"][[7, 2, 5]], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("router", [ROUTER_RENORM, ROUTER_PREK_SOFTMAX, ROUTER_SOFT_GUMBEL])
def test_router_and_expert_parts_equal_the_whole_backward(router):
    # the gate's part and each expert's part on their own (the pieces the
    # full-size GPU checks use) are the whole backward's, value for value;
    # k = 3 of 5 experts over 9 tokens leaves uneven (and maybe empty) experts
    kw = dict(E=5, k=5, pre_k=5, tau=0.8) if router == ROUTER_SOFT_GUMBEL else dict(E=5, k=3)
    cfg = _cfg(router, T=9, **kw)
    a = _inputs(cfg, 11)
    fwd = _exact_forward(cfg, a)
    dout = np.random.default_rng(12).standard_normal((cfg.T, cfg.d))
    whole = oracle.backward(cfg, a, fwd, dout, h_storage="exact")
    part = oracle.backward_router(cfg, a, fwd, dout)
    for n in ("dw", "dL", "dWg", "dbias"):
        np.testing.assert_allclose(part[n], whole[n], rtol=1e-12, atol=1e-14, err_msg=n)
    for e in range(cfg.E):
        pe = oracle.backward_expert(cfg, a, fwd, dout, e, h_storage="exact")
        np.testing.assert_allclose(pe["dW1"], whole["dW1"][e], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(pe["dW2"], whole["dW2"][e], rtol=1e-12, atol=1e-14)
