"""GPU parity of moe_forward on a seeded sweep of random small layers, each
against the whole-layer oracle: every router (renormalised top-k, top-pre_k
softmax, group-limited, Gumbel soft gating), fp32 and bf16, FP8 payloads
with per-token and static scales, packed and gathered rows, both pair-tile
widths, biased and Zipf-skewed loads (experts left empty), and shapes that
reach each gate kernel (shared-memory, narrow, tiled, tensor-core). Tokens
whose routing fp32 cannot decide (the near-tie protocol) are left out of the
comparison; the same tolerances as the fixed layers."""
import numpy as np
import pytest
import torch

import mixture_experts_routed_gb300 as moe
import oracle
from parity_util import assert_close, out_tolerance, route_ties, to_np
from workloads import MoEConfig, make_inputs

pytestmark = pytest.mark.gpu


def _random_layer(i):
    rng = np.random.default_rng(1000 + i)
    dtype = "f32" if rng.random() < 0.2 else "bf16"
    router = int(rng.choice([0, 1, 2, 3], p=[0.4, 0.2, 0.25, 0.15]))
    E = int(rng.choice([1, 3, 8, 16, 24, 32, 40, 64, 128, 256] if router != 3 else [2, 4, 8, 16]))
    d = int(rng.choice([64, 128, 192, 256, 512, 1024]))
    f = int(rng.choice([64, 128, 320, 448, 512]))
    T = int(rng.choice([1, 7, 64, 129, 200, 300]))
    kw = dict(T=T, d=d, E=E, f=f, dtype=dtype, router=router, seed=int(rng.integers(1 << 20)))
    if router == 3:
        kw.update(k=E, pre_k=min(8, E), tau=float(rng.choice([0.5, 1.0, 2.0])))
    else:
        pre_k = int(rng.integers(1, min(8, E) + 1))
        k = int(rng.integers(1, pre_k + 1))
        kw.update(k=k, pre_k=pre_k)
        if router == 2:
            groups = [g for g in (1, 2, 4, 8, 16, 32) if E % g == 0 and g <= E]
            n_group = int(rng.choice(groups))
            need = -(-k // (E // n_group))                # groups needed to hold k experts
            kw.update(n_group=n_group, topk_group=int(rng.integers(need, n_group + 1)))
        if dtype == "bf16" and rng.random() < 0.25:
            static = rng.random() < 0.4
            kw.update(payload_fp8=2 if static else 1, payload_scale=0.02 if static else 0.0,
                      outlier_rate=0.01)
        elif dtype == "bf16" and rng.random() < 0.3:
            kw.update(x_perm_mode=2)
    if dtype == "bf16":
        kw.update(gemm_tile_n=int(rng.choice([0, 256, 512])))
    b = rng.random()
    if b < 0.3:
        kw.update(bias="zipf", zipf_s=1.1)
    elif b < 0.6:
        kw.update(bias="normal", bias_var=0.5)
    return MoEConfig(f"random{i}", **kw)


@pytest.mark.parametrize("i", range(64))
def test_random_layer_matches_oracle(cuda_ok, i):
    cfg = _random_layer(i)
    assert moe.check_config(cfg) == moe.MOE_OK, cfg
    inp = make_inputs(cfg, device="cuda")
    ws = moe.alloc_workspace(cfg)
    out = moe.forward(cfg, inp["x"], inp["Wg"], inp["bias"], inp["W1"], inp["W2"], ws=ws,
                      noise=inp.get("gumbel"))
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == moe.MOE_OK, cfg
    host = oracle.inputs_to_numpy(inp)
    ref = oracle.forward(cfg, host, keep_h=False)
    L = oracle.gate_logits(host["x"], host["Wg"], host["bias"])
    keep = ~route_ties(cfg, L)
    rel, mabs = out_tolerance(cfg)
    assert_close(to_np(out)[keep], ref["out_rounded"][keep], rel, mabs, str(cfg))
    if keep.all():
        v = moe.forward_views(cfg, ws)
        assert np.array_equal(to_np(v["counts"]), ref["counts"]), cfg
        assert np.array_equal(to_np(v["pos"]), ref["pos"]), cfg


def _close(got, ref, rel, what):
    err = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    mabs = np.abs(got - ref).max() if ref.size else 0.0
    scale = np.abs(ref).max() if ref.size else 0.0
    assert err <= rel and mabs <= 10 * rel * max(scale, 1e-30), (what, err, mabs, scale)


@pytest.mark.parametrize("i", range(24))
def test_random_layer_backward_matches_oracle(cuda_ok, i):
    # the FP8 payloads have no backward: the same sweep without them; every
    # other layer's forward keeps Z for the backward
    cfg = _random_layer(100 + i).with_(payload_fp8=0, payload_scale=0.0, outlier_rate=0.0,
                                       keep_z=i % 2)
    assert moe.check_config(cfg) == moe.MOE_OK, cfg
    inp = make_inputs(cfg, device="cuda")
    ws = moe.alloc_workspace(cfg)
    moe.forward(cfg, inp["x"], inp["Wg"], inp["bias"], inp["W1"], inp["W2"], ws=ws,
                noise=inp.get("gumbel"))
    g = torch.Generator(device="cuda")
    g.manual_seed(7 + i)
    dout = torch.randn((cfg.T, cfg.d), generator=g, device="cuda").to(cfg.torch_dtype)
    bws = moe.alloc_workspace(cfg, "backward")
    grads = moe.backward(cfg, inp["x"], inp["Wg"], inp["bias"], inp["W1"], inp["W2"], dout,
                         fwd_ws=ws, ws=bws, noise=inp.get("gumbel"))
    torch.cuda.synchronize()
    assert moe.get_device_error(bws) == moe.MOE_OK and moe.get_device_error(ws) == moe.MOE_OK
    host = oracle.inputs_to_numpy(inp)
    ref_f = oracle.forward(cfg, host)
    L = oracle.gate_logits(host["x"], host["Wg"], host["bias"])
    if route_ties(cfg, L).any():
        pytest.skip("a near-tie token: the routing (and so every gradient) may differ")
    assert np.array_equal(to_np(moe.forward_views(cfg, ws)["topk_idx"]), ref_f["topk_idx"])
    ref = oracle.backward(cfg, host, ref_f, dout.float().cpu().numpy())
    rel = 1e-4 if cfg.dtype == "f32" else 2e-3
    for n in ("dx", "dWg", "dbias", "dW1", "dW2"):
        _close(grads[n].cpu().numpy().astype(np.float64), ref[n], rel, f"{cfg} {n}")


@pytest.mark.parametrize("i", range(12))
def test_random_layer_fp8_expert_outputs_match_oracle(cuda_ok, i):
    # the same sweep with the expert outputs handed to the combine as the FP8
    # min/max-affine payload (hard routers), with its own comparator
    from parity_util import assert_close_output_fp8
    cfg = _random_layer(200 + i)
    if cfg.router == 3:
        cfg = cfg.with_(router=0, k=min(2, cfg.E), pre_k=min(8, cfg.E))
    cfg = cfg.with_(output_fp8=1)
    assert moe.check_config(cfg) == moe.MOE_OK, cfg
    inp = make_inputs(cfg, device="cuda")
    ws = moe.alloc_workspace(cfg)
    out = moe.forward(cfg, inp["x"], inp["Wg"], inp["bias"], inp["W1"], inp["W2"], ws=ws,
                      noise=inp.get("gumbel"))
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == moe.MOE_OK, cfg
    host = oracle.inputs_to_numpy(inp)
    ref = oracle.forward(cfg, host, keep_h=False)
    L = oracle.gate_logits(host["x"], host["Wg"], host["bias"])
    keep = ~route_ties(cfg, L)
    slots = ref["pos"].reshape(cfg.T, cfg.k)
    v = moe.forward_views(cfg, ws)
    rows = torch.from_numpy(slots.reshape(-1).astype(np.int64)).cuda()
    codes = v["y_q"][rows].view(torch.float8_e4m3fn).double().cpu().numpy()
    codes = codes.reshape(cfg.T, cfg.k, -1)
    assert_close_output_fp8(cfg, to_np(out)[keep], ref["out_rounded"][keep], ref["topk_w"][keep],
                            ref["y_q"][slots][keep], ref["y_scale"][slots][keep], codes[keep],
                            str(cfg))
