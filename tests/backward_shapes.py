"""Backward parity shapes (small layers for every router mode, fp32 and
bf16, a single expert, experts with no rows, ragged batches and tiles partly
past the matrix edge), shared by the GPU parity tests and the CPU check that
each is a valid layer the oracle can differentiate."""
from workloads import MoEConfig, ROUTER_GROUP_LIMITED, ROUTER_PREK_SOFTMAX, \
    ROUTER_SOFT_GUMBEL, get_config

SHAPES = {
    "bwd_bf16_T129_d256_E8_k2_f320": MoEConfig(
        "bwd_bf16_T129_d256_E8_k2_f320", T=129, d=256, E=8, k=2, f=320, dtype="bf16",
        bias="normal", bias_var=0.5, seed=70),
    "bwd_f32_T50_d64_E5_k2_f128": MoEConfig(
        "bwd_f32_T50_d64_E5_k2_f128", T=50, d=64, E=5, k=2, f=128, dtype="f32", pre_k=5,
        seed=71),
    "bwd_prek_T200_d256_E64_k2_f128": MoEConfig(
        "bwd_prek_T200_d256_E64_k2_f128", T=200, d=256, E=64, k=2, f=128, dtype="bf16",
        router=ROUTER_PREK_SOFTMAX, bias="normal", bias_var=0.5, seed=72),
    "bwd_group_T300_d256_E16_k2_f128": MoEConfig(
        "bwd_group_T300_d256_E16_k2_f128", T=300, d=256, E=16, k=2, f=128, dtype="bf16",
        router=ROUTER_GROUP_LIMITED, n_group=4, topk_group=2, seed=73),
    "bwd_soft_T100_d256_E8_f128": MoEConfig(
        "bwd_soft_T100_d256_E8_f128", T=100, d=256, E=8, k=8, f=128, dtype="bf16",
        router=ROUTER_SOFT_GUMBEL, tau=0.7, seed=74),
    "bwd_soft_f32_T64_d128_E4_f128": MoEConfig(
        "bwd_soft_f32_T64_d128_E4_f128", T=64, d=128, E=4, k=4, f=128, dtype="f32", pre_k=4,
        router=ROUTER_SOFT_GUMBEL, tau=1.0, seed=75),
    "bwd_single_T70_d128_E1_k1_f192": MoEConfig(
        "bwd_single_T70_d128_E1_k1_f192", T=70, d=128, E=1, k=1, f=192, dtype="bf16", pre_k=1,
        seed=76),
    "bwd_skew_T256_d128_E64_k8_f128_zipf": MoEConfig(
        "bwd_skew_T256_d128_E64_k8_f128_zipf", T=256, d=128, E=64, k=8, f=128, dtype="bf16",
        bias="zipf", zipf_s=3.0, seed=77),
    "bwd_tiny_fp32_layer": get_config("tiny_T256_d128_E8_k2_f256_fp32"),
    # one token: most experts have no rows
    "bwd_one_token_T1_d64_E4_k2_f64": MoEConfig(
        "bwd_one_token_T1_d64_E4_k2_f64", T=1, d=64, E=4, k=2, f=64, dtype="bf16", pre_k=4,
        seed=78),
    # d = 192, f = 448: pair tiles whose odd half is partly or wholly past M / N
    "bwd_ragged_T96_d192_E3_k2_f448": MoEConfig(
        "bwd_ragged_T96_d192_E3_k2_f448", T=96, d=192, E=3, k=2, f=448, dtype="bf16",
        pre_k=3, seed=79),
    # E = 128: both gate GEMMs on the tensor cores; experts of a few rows
    "bwd_gate_tc_T160_d128_E128_k4_f64": MoEConfig(
        "bwd_gate_tc_T160_d128_E128_k4_f64", T=160, d=128, E=128, k=4, f=64, dtype="bf16",
        bias="normal", bias_var=0.5, seed=80),
    # a single expert of exactly 128 rows (whole 64-row blocks, no tail)
    "bwd_whole_blocks_T128_d128_E1_k1_f128": MoEConfig(
        "bwd_whole_blocks_T128_d128_E1_k1_f128", T=128, d=128, E=1, k=1, f=128,
        dtype="bf16", pre_k=1, seed=81),
}
