"""Figures printed on the source pages, reproduced by the oracle and by the
host-side load statistics (CPU only). Fixture: tests/golden/page_figures.json."""
import json
import os

import numpy as np

import oracle
from mixture_experts_routed_gb300.stats import load_stats

FIX = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))


def test_routing_index_array_is_8_kb():
    f = FIX["routing_index_bytes"]
    rng = np.random.default_rng(0)
    L = rng.standard_normal((f["T"], 8))
    idx, _ = oracle.route(L, f["k"])
    assert idx.dtype == np.int32 and idx.shape == (f["T"], f["k"])
    assert idx.nbytes == f["bytes"]


def test_ideal_activation_rate():
    f = FIX["ideal_activation_rate"]
    s = load_stats([10] * f["E"])
    assert round(100 * s["ideal_share"], 2) == f["percent_2dp"]
    assert s["max_share"] == s["min_share"] == s["ideal_share"]


def test_ideal_entropy_and_skew():
    f = FIX["ideal_routing_entropy"]
    s = load_stats([7] * f["E"])
    assert s["entropy_bits"] == f["bits"] == s["ideal_entropy_bits"]
    skew = load_stats([100] + [1] * (f["E"] - 1))
    assert skew["entropy_bits"] < f["bits"]
    assert skew["max_over_mean"] > 10
    s0 = load_stats([4, 0, 0, 4])
    assert s0["zero_experts"] == 2 and s0["entropy_bits"] == 1.0


def test_fp8_payload_size():
    f = FIX["fp8_payload_halves_fp16"]
    x = np.random.default_rng(1).standard_normal((16, 64))
    q, s = oracle.quantize_payload_fp8(x)
    payload = oracle.e4m3_encode(q)
    assert payload.dtype == np.uint8
    assert payload.nbytes * f["fp16_bytes_per_elem"] == x.astype(np.float16).nbytes * f["fp8_bytes_per_elem"]
