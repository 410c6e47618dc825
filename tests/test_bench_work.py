"""The algorithmic bytes and flops bench.py divides by a kernel's time (the
numerator of every roofline fraction it prints), against figures worked out
by hand from the kernel table's formulas: every operand read once, every
result written once, weights only of experts that received rows. The
skewed 256-expert layer's figures are the byte counts its bench line reports
(211 of 256 experts receive rows under its seeded Zipf load)."""
import bench
from workloads import get_config

SKEWED = "skewed_T16384_d7168_E256_k8_f2048_zipf"
BALANCED = "balanced_T1024_d4096_E8_k2_f11008"
WIDE_FP8 = "wide_fp8_T16384_d5120_E16_k2_f1536"


def _counts(E, active):
    return [1] * active + [0] * (E - active)


def test_skewed_layer_gathered_rows():
    w = bench.stage_work(get_config(SKEWED), _counts(256, 211), gathered=True)
    # T d b + d E b + 4 E + 8 R = 234881024 + 3670016 + 1024 + 1048576
    assert w["route"] == (239_600_640, 60_129_542_144.0)
    # only the layout: 12 R + 8 E
    assert w["dispatch"] == (1_574_912, 0.0)
    # A d f b + R d b + R f b = 6194987008 + 1879048192 + 536870912
    assert w["gemm_w1_silu"] == (8_610_906_112, 3_848_290_697_216.0)
    # A f d b + R f b + 4 R d = 6194987008 + 536870912 + 3758096384
    assert w["gemm_w2"] == (10_489_954_304, 3_848_290_697_216.0)
    # 4 R d + 8 R + T d b = 3758096384 + 1048576 + 234881024
    assert w["combine"] == (3_994_025_984, 1_879_048_192.0)
    assert w["quantize_out"] == (0, 0.0)


def test_skewed_layer_packed_rows_dispatch():
    w = bench.stage_work(get_config(SKEWED), _counts(256, 211), gathered=False)
    # T d b + R d b + 12 R = 234881024 + 1879048192 + 1572864
    assert w["dispatch"] == (2_115_502_080, 0.0)
    assert w["gemm_w1_silu"][0] == 8_610_906_112


def test_balanced_layer_w1():
    w = bench.stage_work(get_config(BALANCED), _counts(8, 8))
    # 8 d f b + R d b + R f b = 721420288 + 16777216 + 45088768
    assert w["gemm_w1_silu"] == (783_286_272, 2.0 * 2048 * 4096 * 11008)
    # an expert without rows moves none of its weights
    w7 = bench.stage_work(get_config(BALANCED), _counts(8, 7))
    assert w["gemm_w1_silu"][0] - w7["gemm_w1_silu"][0] == 4096 * 11008 * 2
    assert w["gemm_w2"][0] - w7["gemm_w2"][0] == 4096 * 11008 * 2


def test_fp8_payload_layer():
    w = bench.stage_work(get_config(WIDE_FP8), _counts(16, 16))
    # T d b + R d (one byte per E4M3 code) + 12 R + 4 R (scales)
    # = 167772160 + 167772160 + 393216 + 131072
    assert w["dispatch"] == (336_068_608, 0.0)
    # 16 d f b + R d + R f b = 251658240 + 167772160 + 100663296
    assert w["gemm_w1_silu"][0] == 520_093_696


def test_fp32_layer_counts_four_bytes():
    c = get_config("tiny_T256_d128_E8_k2_f256_fp32")
    w = bench.stage_work(c, _counts(8, 8))
    # 8 f d 4 + R f 4 + 4 R d = 1048576 + 524288 + 262144
    assert w["gemm_w2"] == (1_835_008, 2.0 * 512 * 256 * 128)
