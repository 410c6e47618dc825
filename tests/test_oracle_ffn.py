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
