"""The seeded input generator (CPU only): determinism and the recipe.

Re-drawing a shape with its seed gives identical bytes; a different seed does
not; the draws follow the stated distributions (x ~ N(0, 1), W_g and W1 ~
N(0, 1/d), W2 ~ N(0, 1/f), the normal gate bias's variance, the +-20
outliers at their rate, the Zipf bias as -s ln(rank) over a permutation, the
Gumbel samples' mean and variance) and the layer dtypes."""
import hashlib
import math

import numpy as np
import torch

from workloads import CONFIGS, VARIANTS, get_config, make_inputs


def _digest(inp):
    h = hashlib.sha256()
    for k in sorted(inp):
        h.update(k.encode())
        h.update(inp[k].contiguous().view(torch.uint8).numpy().tobytes())
    return h.hexdigest()


def _small(name, **kw):
    base = dict(T=512, d=256, f=128)
    base.update(kw)
    return get_config(name).with_(**base)


def test_same_seed_same_bytes_other_seed_other_bytes():
    for name in ("balanced_T1024_d4096_E8_k2_f11008", "wide_fp8_T16384_d5120_E16_k2_f1536",
                 "soft_gumbel_T16384_d5120_E16_f1536"):
        cfg = _small(name)
        assert _digest(make_inputs(cfg)) == _digest(make_inputs(cfg))
        assert _digest(make_inputs(cfg)) != _digest(make_inputs(cfg.with_(seed=cfg.seed + 1)))


def test_distributions_and_dtypes():
    cfg = _small("balanced_T1024_d4096_E8_k2_f11008", T=2048, d=512, f=256)
    a = make_inputs(cfg)
    assert a["x"].dtype == torch.bfloat16 and a["W1"].dtype == torch.bfloat16
    assert a["bias"].dtype == torch.float32 and not torch.any(a["bias"])
    for key, std in (("x", 1.0), ("Wg", 1 / math.sqrt(cfg.d)), ("W1", 1 / math.sqrt(cfg.d)),
                     ("W2", 1 / math.sqrt(cfg.f))):
        v = a[key].float()
        n = v.numel()
        assert abs(v.mean().item()) < 5 * std / math.sqrt(n), key
        assert abs(v.std().item() / std - 1) < 0.02, key
    tiny = make_inputs(get_config("tiny_T256_d128_E8_k2_f256_fp32"))
    assert tiny["x"].dtype == torch.float32 and tiny["W2"].dtype == torch.float32


def test_normal_bias_variance():
    cfg = get_config("many_expert_T8192_d2048_E64_k2_f1408_prek8").with_(T=8, d=64, f=64, E=256)
    b = np.concatenate([make_inputs(cfg.with_(seed=s))["bias"].numpy() for s in range(40)])
    assert abs(b.var() / 0.5 - 1) < 0.05


def test_outliers_rate_and_value():
    cfg = _small("wide_fp8_T16384_d5120_E16_k2_f1536", T=1024, d=1024)
    x = make_inputs(cfg)["x"].float()
    hit = x.abs() == 20.0
    n = x.numel()
    rate = hit.float().mean().item()
    assert abs(rate - 1e-3) < 5 * math.sqrt(1e-3 / n)
    # both signs, about equally often
    pos = (x[hit] > 0).float().mean().item()
    assert 0.35 < pos < 0.65


def test_zipf_bias_is_minus_s_log_rank_over_a_permutation():
    cfg = get_config("skewed_T16384_d7168_E256_k8_f2048_zipf").with_(T=8, d=64, f=64)
    b = make_inputs(cfg)["bias"].numpy().astype(np.float64)
    expect = -1.1 * np.log(np.arange(1, cfg.E + 1))
    np.testing.assert_allclose(np.sort(b)[::-1], expect, rtol=0, atol=1e-6)
    assert b.argmax() != 0 or b.argmin() != cfg.E - 1     # not left in rank order


def test_gumbel_samples():
    cfg = _small("soft_gumbel_T16384_d5120_E16_f1536", T=8192)
    g = make_inputs(cfg)["gumbel"].double()
    assert g.shape == (cfg.T, cfg.E)
    n = g.numel()
    assert abs(g.mean().item() - 0.5772156649) < 5 * (math.pi / math.sqrt(6)) / math.sqrt(n)
    assert abs(g.var().item() / (math.pi ** 2 / 6) - 1) < 0.03


def test_every_named_shape_is_a_valid_config():
    import mixture_experts_routed_gb300 as moe
    for cfg in list(CONFIGS.values()) + list(VARIANTS.values()):
        assert moe.check_config(cfg) == 0, cfg.name
