"""moe_dispatch_noalloc: the dispatch for callers that cannot allocate device
memory (its scratch tables live in a fixed array inside the library instead
of a caller workspace). Checked through the C ABI against moe_dispatch on
two calls in a row, so a second call cannot pick up anything the first left
in the shared array. This file is collected last; it builds the library and
draws its own inputs, so it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_routed_gb300 import _lib as L
from mixture_experts_routed_gb300 import build as B
from workloads import MoEConfig, make_inputs

pytestmark = pytest.mark.gpu

SHAPES = [
    MoEConfig("na_bf16_T129_d256_E8_k2", T=129, d=256, E=8, k=2, f=128, dtype="bf16", seed=31),
    MoEConfig("na_fp8_T300_d512_E16_k2", T=300, d=512, E=16, k=2, f=128, dtype="bf16",
              payload_fp8=True, outlier_rate=0.01, seed=32),
    # one static FP8 scale for every row (small enough that the outliers saturate)
    MoEConfig("na_fp8static_T300_d512_E16_k2", T=300, d=512, E=16, k=2, f=128, dtype="bf16",
              payload_fp8=2, payload_scale=0.02, outlier_rate=0.01, seed=35),
    MoEConfig("na_f32_T64_d128_E5_k2", T=64, d=128, E=5, k=2, f=128, dtype="f32", pre_k=5,
              seed=33),
    MoEConfig("na_zipf_T2048_d256_E256_k8", T=2048, d=256, E=256, k=8, f=128, dtype="bf16",
              bias="zipf", zipf_s=1.1, seed=34),
]


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    return L.load()


def _cfg(c):
    return L.MoeConfig(c.T, c.d, c.E, c.k, c.f, 0 if c.dtype == "f32" else 1, c.router,
                       c.pre_k, int(c.payload_fp8), payload_scale=c.payload_scale)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _outputs(c):
    R = c.T * c.k
    i32 = dict(dtype=torch.int32, device="cuda")
    pdt = torch.uint8 if c.payload_fp8 else (torch.float32 if c.dtype == "f32" else torch.bfloat16)
    return {"counts": torch.full((c.E,), -9, **i32), "offsets": torch.full((c.E + 1,), -9, **i32),
            "pos": torch.full((R,), -9, **i32), "src": torch.full((R,), -9, **i32),
            "x_perm": torch.zeros((R, c.d), dtype=pdt, device="cuda"),
            "x_scale": torch.zeros(R, dtype=torch.float32, device="cuda") if c.payload_fp8 else None}


def _routing(lib, c, inp):
    cc = _cfg(c)
    idx = torch.empty((c.T, c.k), dtype=torch.int32, device="cuda")
    w = torch.empty((c.T, c.k), dtype=torch.float32, device="cuda")
    st = lib.moe_route(ctypes.byref(cc), _p(inp["x"]), _p(inp["Wg"]), _p(inp["bias"]), None,
                       _p(idx), _p(w), None,
                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == L.MOE_OK
    return idx


def _with_workspace(lib, c, x, idx):
    cc = _cfg(c)
    o = _outputs(c)
    n = lib.moe_scratch_size(ctypes.byref(cc))
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    st = lib.moe_dispatch(ctypes.byref(cc), _p(x), _p(idx), _p(o["counts"]), _p(o["offsets"]),
                          _p(o["pos"]), _p(o["src"]), _p(o["x_perm"]), _p(o["x_scale"]), _p(ws),
                          n, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == L.MOE_OK
    return o


def _without_workspace(lib, c, x, idx):
    cc = _cfg(c)
    o = _outputs(c)
    st = lib.moe_dispatch_noalloc(ctypes.byref(cc), _p(x), _p(idx), _p(o["counts"]),
                                  _p(o["offsets"]), _p(o["pos"]), _p(o["src"]),
                                  _p(o["x_perm"]), _p(o["x_scale"]),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == L.MOE_OK
    return o


def _same(a, b):
    for key in ("counts", "offsets", "pos", "src", "x_perm", "x_scale"):
        if a[key] is None:
            assert b[key] is None
            continue
        assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("c", SHAPES, ids=[c.name for c in SHAPES])
def test_noalloc_dispatch_matches_dispatch_on_two_calls(lib, c):
    # two different batches in a row through the shared scratch array
    for shift in (0, 1):
        inp = make_inputs(c.with_(seed=c.seed + 100 * shift), device="cuda")
        idx = _routing(lib, c, inp)
        ref = _with_workspace(lib, c, inp["x"], idx)
        got = _without_workspace(lib, c, inp["x"], idx)
        torch.cuda.synchronize()
        _same(ref, got)
        assert int(got["offsets"][-1]) == c.T * c.k


def test_noalloc_dispatch_rejects_oversized_requests(lib):
    c = MoEConfig("na_big", T=16392, d=128, E=256, k=8, f=128, dtype="bf16")
    cc = _cfg(c)
    fake = ctypes.c_void_p(1 << 20)
    st = lib.moe_dispatch_noalloc(ctypes.byref(cc), fake, fake, fake, fake, fake, fake, fake,
                                  None, None)
    assert st == L.MOE_ERR_WORKSPACE_TOO_SMALL
    ok = MoEConfig("na_edge", T=16384, d=128, E=256, k=8, f=128, dtype="bf16")
    assert lib.moe_check_config(ctypes.byref(_cfg(ok))) == L.MOE_OK
