"""Pins for the oracle's expert FFN, combine and whole-layer forward (CPU).

Independent references: torch fp64 dense FFN (matmul + torch's SiLU),
pure-Python loops for the combine, and special cases with closed forms
(one expert, identical experts, linearity in W2)."""
import numpy as np
import pytest
import torch

import oracle
from workloads import MoEConfig, make_inputs, ROUTER_PREK_SOFTMAX


def _cfg(**kw):
    base = dict(name="t", T=37, d=64, E=4, k=2, f=128, dtype="f32", seed=5)
    base.update(kw)
    return MoEConfig(**base)


def _torch_dense_ffn(x, W1, W2, h_round=None):
    z = torch.from_numpy(x) @ torch.from_numpy(W1)
    h = torch.nn.functional.silu(z)
    if h_round == "f32":
        h = h.float().double()
    elif h_round == "bf16":
        h = h.to(torch.bfloat16).double()
    return (h @ torch.from_numpy(W2)).numpy()


def test_one_expert_is_a_dense_ffn():
    cfg = _cfg(E=1, k=1)
    inp = make_inputs(cfg)
    r = oracle.forward(cfg, inp)
    a = oracle.inputs_to_numpy(inp)
    ref = _torch_dense_ffn(a["x"], oracle.moe_oracle._expert(a["W1"], 0),
                           oracle.moe_oracle._expert(a["W2"], 0), "f32")
    assert np.all(r["topk_w"] == 1.0)
    assert np.max(np.abs(r["out"] - ref)) <= 1e-12


def test_one_expert_bf16_storage_of_h():
    cfg = _cfg(E=1, k=1, dtype="bf16")
    inp = make_inputs(cfg)
    r = oracle.forward(cfg, inp)
    a = oracle.inputs_to_numpy(inp)
    ref = _torch_dense_ffn(a["x"], oracle.moe_oracle._expert(a["W1"], 0),
                           oracle.moe_oracle._expert(a["W2"], 0), "bf16")
    # torch rounds the fp64 SiLU to bf16 directly, as the oracle does
    assert np.max(np.abs(r["out"] - ref)) <= 1e-12


@pytest.mark.parametrize("router", [0, ROUTER_PREK_SOFTMAX])
def test_identical_experts_give_ffn_times_weight_sum(router):
    cfg = _cfg(E=5, k=2, router=router, pre_k=4, bias="normal", bias_var=1.0)
    inp = make_inputs(cfg)
    inp["W1"][:] = inp["W1"][0]
    inp["W2"][:] = inp["W2"][0]
    r = oracle.forward(cfg, inp)
    a = oracle.inputs_to_numpy(inp)
    ffn = _torch_dense_ffn(a["x"], oracle.moe_oracle._expert(a["W1"], 0),
                           oracle.moe_oracle._expert(a["W2"], 0), "f32")
    wsum = r["topk_w"].sum(1, keepdims=True)
    assert np.max(np.abs(r["out"] - ffn * wsum)) <= 1e-12
    if router == 0:
        assert np.max(np.abs(wsum - 1.0)) <= 1e-12
    else:
        assert np.all(wsum < 1.0)


def test_linear_in_w2():
    cfg = _cfg()
    inp = make_inputs(cfg)
    r1 = oracle.forward(cfg, inp)
    inp2 = dict(inp)
    inp2["W2"] = inp["W2"] * 2
    r2 = oracle.forward(cfg, inp2)
    assert np.array_equal(r2["out"], 2 * r1["out"])


def test_combine_matches_loops():
    rng = np.random.default_rng(3)
    T, k, d = 6, 3, 5
    R = T * k
    Y = rng.standard_normal((R, d))
    pos = rng.permutation(R)
    w = rng.random((T, k))
    out = oracle.combine(Y, pos, w)
    for t in range(T):
        for c in range(d):
            s = 0.0
            for j in range(k):
                s += w[t, j] * Y[pos[t * k + j], c]
            assert abs(out[t, c] - s) <= 1e-14


def test_forward_tokens_agrees_with_forward():
    cfg = _cfg(T=50, E=6, k=3, dtype="bf16", bias="normal", bias_var=0.5)
    inp = make_inputs(cfg)
    full = oracle.forward(cfg, inp)
    toks = [0, 7, 13, 49]
    part = oracle.forward_tokens(cfg, inp, toks)
    assert np.array_equal(part["topk_idx"], full["topk_idx"][toks])
    assert np.max(np.abs(part["out"] - full["out"][toks])) <= 1e-12


def test_fp8_payload_forward():
    cfg = _cfg(T=40, d=128, dtype="bf16", payload_fp8=True, outlier_rate=0.01)
    inp = make_inputs(cfg)
    r = oracle.forward(cfg, inp)
    a = oracle.inputs_to_numpy(inp)
    # the experts see q*s of the token's own row, one scale per token
    q_tok, s_tok = oracle.quantize_payload_fp8(a["x"])
    assert np.array_equal(r["q"], q_tok[r["src"]])
    assert np.array_equal(r["scale"], s_tok[r["src"]])
    # quantisation moves the output, but only by a bounded amount
    plain = oracle.forward(cfg.with_(payload_fp8=False), inp)
    rel = np.linalg.norm(r["out"] - plain["out"]) / np.linalg.norm(plain["out"])
    assert 1e-4 < rel < 0.1


def test_empty_expert_does_not_contribute():
    cfg = _cfg(E=6, k=1)
    inp = make_inputs(cfg)
    inp["bias"] = torch.tensor([0, 0, 0, -1e4, 0, 0], dtype=torch.float32)
    r = oracle.forward(cfg, inp)
    assert r["counts"][3] == 0
    inp["W1"][3] = float("nan")                 # never read
    r2 = oracle.forward(cfg, inp)
    assert np.array_equal(r["out"], r2["out"])


@pytest.mark.parametrize("f_extra", [0, 64])
def test_permutation_weights_give_scaled_silu(f_extra):
    # W1_e = [P_e | 0] (d x f), W2_e = c_e [P_e^T ; R] (f x d): row-vector
    # convention x W1 permutes x, SiLU acts elementwise (SiLU(0) = 0 on the
    # padding columns, so R never matters), W2 undoes the permutation. So
    # expert e returns c_e SiLU(x) exactly and the layer returns
    # (sum_j w_tj c_e(t,j)) SiLU(x_t), checked with math.exp. A transposed or
    # mis-indexed W1 or W2, or a combine using the wrong expert's output,
    # fails this.
    import math
    d, E, k = 64, 6, 3
    cfg = _cfg(d=d, E=E, k=k, f=d + f_extra, pre_k=4, bias="normal", bias_var=1.0)
    inp = make_inputs(cfg)
    a = oracle.inputs_to_numpy(inp)
    rng = np.random.default_rng(11)
    c = rng.uniform(0.5, 2.0, size=E)
    W1 = np.zeros((E, d, cfg.f))
    W2 = rng.standard_normal((E, cfg.f, d))       # rows past d are multiplied by SiLU(0) = 0
    for e in range(E):
        P = np.eye(d)[rng.permutation(d)]
        W1[e, :, :d] = P
        W2[e, :d, :] = c[e] * P.T
    a["W1"], a["W2"] = W1, W2
    r = oracle.forward(cfg, a)
    x = a["x"]
    # H is stored in the layer's dtype (fp32 here), so SiLU(x) is rounded to fp32
    silu = np.vectorize(lambda v: v / (1.0 + math.exp(-v)))(x).astype(np.float32).astype(np.float64)
    scale = np.array([sum(r["topk_w"][t, j] * c[r["topk_idx"][t, j]] for j in range(k))
                      for t in range(cfg.T)])
    assert np.max(np.abs(r["out"] - scale[:, None] * silu)) <= 1e-12


@pytest.mark.parametrize("mistake", ["w1_transposed", "w2_transposed", "no_silu", "wrong_expert"])
def test_permutation_pin_catches_planted_mistakes(monkeypatch, mistake):
    # the pin above must fail when the oracle's FFN is wrong in a plausible
    # way: a mistake planted in the oracle (on the CPU) is caught
    mo = oracle.moe_oracle
    real_rows, real_expert = mo.expert_ffn_rows, mo._expert

    def bad_rows(x_rows, W1e, W2e, h_storage="bf16"):
        # (the pin runs with f = d here, so the weights are square)
        if mistake == "w1_transposed":
            return real_rows(x_rows, np.asarray(W1e).T, W2e, h_storage)
        if mistake == "w2_transposed":
            return real_rows(x_rows, W1e, np.asarray(W2e).T, h_storage)
        if mistake == "no_silu":
            z = np.asarray(x_rows, np.float64) @ np.asarray(W1e, np.float64)
            h = mo.round_to_f32(z) if h_storage == "f32" else z
            return h @ np.asarray(W2e, np.float64), h
        return real_rows(x_rows, W1e, W2e, h_storage)

    def bad_expert(W, e):
        return real_expert(W, (e + 1) % W.shape[0]) if mistake == "wrong_expert" else real_expert(W, e)

    monkeypatch.setattr(mo, "expert_ffn_rows", bad_rows)
    monkeypatch.setattr(mo, "_expert", bad_expert)
    with pytest.raises(AssertionError):
        test_permutation_weights_give_scaled_silu(0)
