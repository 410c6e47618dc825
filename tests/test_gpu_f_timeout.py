"""The bounded-wait path of the grouped expert GEMM, run on the GPU.

Every wait in the library's kernels gives up after a bound, flags
MOE_ERR_TIMEOUT and lets the kernel finish cleanly. Here a test hook
shortens one such bound, the GEMM epilogue's wait for a finished
accumulator, to 1 ns, so that it runs out on the first tile (the device
timer ticks in far less than a tile's main loop on these layers): the forward
must come back (within the other waits' own 2 s bounds) with
MOE_ERR_TIMEOUT, and the context must stay usable: the same forward run
afterwards with the default bound gives the bits of a run made before.
Nothing is left to hang: no flag is waited on that nothing sets except
through the bound, and no copy or tensor-core instruction is abandoned."""
import time

import pytest
import torch

import mixture_experts_routed_gb300 as moe
from mixture_experts_routed_gb300 import _lib as L
from workloads import get_config, make_inputs

pytestmark = pytest.mark.gpu

# Layers with long contractions (d = 5120, 7168: a tile's main loop takes tens
# of microseconds, far longer than the device timer's resolution, so a 1 ns
# bound runs out on the first tile): the 2048-token copy of the 256-expert
# shape with packed rows, gathered rows and 512-feature tiles (one
# accumulator), and 512 tokens of the FP8-payload layer (the row converters).
SMALL_SKEWED = "skewed_small_T2048_d7168_E32_k8_f2048_zipf"
CASES = [(SMALL_SKEWED, moe.MOE_XPERM_PACKED, 0, None),
         (SMALL_SKEWED, moe.MOE_XPERM_GATHERED, 0, None),
         (SMALL_SKEWED, moe.MOE_XPERM_PACKED, 512, None),
         ("wide_fp8_T16384_d5120_E16_k2_f1536", moe.MOE_XPERM_AUTO, 0, 512)]


def _forward(cfg, inp):
    ws = moe.alloc_workspace(cfg)
    out = moe.forward(cfg, inp["x"], inp["Wg"], inp["bias"], inp["W1"], inp["W2"], ws=ws)
    torch.cuda.synchronize()
    return out, moe.get_device_error(ws)


@pytest.mark.parametrize("name,mode,width,tokens", CASES)
def test_gemm_wait_runs_out_and_the_context_stays_usable(cuda_ok, name, mode, width, tokens):
    cfg = get_config(name).with_(x_perm_mode=mode, gemm_tile_n=width)
    if tokens is not None:
        cfg = cfg.with_(T=tokens)
    inp = make_inputs(cfg, device="cuda")
    ref, st = _forward(cfg, inp)
    assert st == moe.MOE_OK
    lib = L.load()
    try:
        assert lib.moe_set_gemm_epilogue_wait_ns(1) == moe.MOE_OK
        t0 = time.monotonic()
        _, st = _forward(cfg, inp)
        elapsed = time.monotonic() - t0
    finally:
        lib.moe_set_gemm_epilogue_wait_ns(0)
    assert st == moe.MOE_ERR_TIMEOUT
    assert elapsed < 30.0
    again, st = _forward(cfg, inp)
    assert st == moe.MOE_OK
    assert torch.equal(again, ref)
    print(f"{cfg.name} mode {mode} width {width}: timed-out forward took {elapsed:.2f} s")
