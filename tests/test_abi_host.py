"""The C-ABI library builds, loads and exports exactly what include/moe.h
declares; host-side validation returns the documented status codes. No test
here reaches a CUDA call (they all fail validation first), so the file runs
without a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

from mixture_experts_routed_gb300 import build as B
from mixture_experts_routed_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.load()


def header_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text))
    return names


def test_header_declares_the_stage_calls():
    names = header_functions()
    for n in ("moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = header_functions()
    assert names == set(L.PROTOTYPES), names ^ set(L.PROTOTYPES)
    for n in names:
        assert getattr(lib, n) is not None


def test_only_abi_symbols_are_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True,
                         text=True).stdout
    funcs = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert header_functions() <= funcs
    stray = {f for f in funcs if not f.startswith("moe_") and not f.startswith("_")}
    assert not stray, stray


def header_source():
    """The headers' text with the comments taken out."""
    text = "".join(open(os.path.join(ROOT, "include", fn)).read()
                   for fn in sorted(os.listdir(os.path.join(ROOT, "include"))) if fn.endswith(".h"))
    return re.sub(r"/\*.*?\*/", " ", text, flags=re.S)


def struct_fields(tag):
    body = re.search(r"typedef struct %s \{(.*?)\}" % tag, header_source(), re.S).group(1)
    fields = []
    for decl in body.split(";"):
        decl = " ".join(decl.split())
        if decl:
            ctype, ptr, name = re.fullmatch(r"([\w ]+?)\s*(\**)\s*(\w+)", decl).groups()
            fields.append((name, ctype + ptr))
    return fields


def test_config_struct_matches_the_header():
    # the ctypes mirror must have the header's fields, in its order and types
    # (a drift would shift every later field of every call)
    fields = struct_fields("moe_config")
    assert [n for n, _ in fields] == [n for n, _ in L.MoeConfig._fields_]
    ctypes_of = {"int32_t": ctypes.c_int32, "float": ctypes.c_float}
    for (name, ctype), (_, mirror) in zip(fields, L.MoeConfig._fields_):
        assert ctypes_of[ctype] is mirror, name
    assert ctypes.sizeof(L.MoeConfig) == 4 * len(fields)


def test_views_struct_matches_the_header():
    fields = struct_fields("moe_forward_views")
    assert [n for n, _ in fields] == [n for n, _ in L.MoeForwardViews._fields_]
    assert all(ctype.endswith("*") for _, ctype in fields)
    assert all(t is ctypes.c_void_p for _, t in L.MoeForwardViews._fields_)


def _param_ctype(param):
    if "moe_config_t*" in param:
        return ctypes.POINTER(L.MoeConfig)
    if "moe_forward_views_t*" in param:
        return ctypes.POINTER(L.MoeForwardViews)
    if param.startswith("void* const*"):
        return ctypes.POINTER(ctypes.c_void_p)
    if "*" in param:
        return ctypes.c_void_p
    kind = param.split()[0]
    return {"size_t": ctypes.c_size_t, "int": ctypes.c_int, "int32_t": ctypes.c_int,
            "uint64_t": ctypes.c_uint64}[kind]


def test_every_prototype_matches_the_header():
    # each function's return type, parameter count and parameter kinds
    # (pointer, size_t, int, uint64_t) against its ctypes prototype
    rets = {"int": ctypes.c_int, "size_t": ctypes.c_size_t, "const char*": ctypes.c_char_p}
    seen = set()
    for m in re.finditer(r"MOE_API\s+([\w\s\*]+?)\b(moe_\w+)\s*\((.*?)\)\s*;",
                         header_source(), re.S):
        ret, name, params = " ".join(m.group(1).split()), m.group(2), " ".join(m.group(3).split())
        res, args = L.PROTOTYPES[name]
        assert rets[ret] is res, name
        plist = [] if params in ("", "void") else [q.strip() for q in params.split(",")]
        assert len(plist) == len(args), name
        for q, a in zip(plist, args):
            assert _param_ctype(q) is a, (name, q)
        seen.add(name)
    assert seen == set(L.PROTOTYPES)


def cfg(**kw):
    base = dict(T=64, d=128, E=8, k=2, f=256, dtype=1, router=0, pre_k=8, payload_fp8=0,
                n_group=0, topk_group=0, payload_scale=0.0, output_fp8=0, tau=0.0,
                gemm_tile_n=0, x_perm_mode=0, keep_z=0)
    base.update(kw)
    return L.MoeConfig(*[base[n] for n, _ in L.MoeConfig._fields_])


@pytest.mark.parametrize("kw,status", [
    ({}, L.MOE_OK),
    (dict(T=0), L.MOE_OK),
    (dict(dtype=0), L.MOE_OK),
    (dict(payload_fp8=1), L.MOE_OK),
    (dict(E=256, k=8), L.MOE_OK),
    (dict(E=1, k=1, pre_k=1), L.MOE_OK),
    (dict(router=1, E=64), L.MOE_OK),
    (dict(T=-1), L.MOE_ERR_INVALID_ARG),
    (dict(d=100), L.MOE_ERR_INVALID_ARG),
    (dict(f=96), L.MOE_ERR_INVALID_ARG),
    (dict(E=0), L.MOE_ERR_INVALID_ARG),
    (dict(E=257), L.MOE_ERR_INVALID_ARG),
    (dict(k=0), L.MOE_ERR_INVALID_ARG),
    (dict(k=9, pre_k=8), L.MOE_ERR_INVALID_ARG),
    (dict(k=3, pre_k=2), L.MOE_ERR_INVALID_ARG),
    (dict(E=4, k=2, pre_k=8), L.MOE_ERR_INVALID_ARG),
    (dict(dtype=2), L.MOE_ERR_INVALID_ARG),
    # group-limited router: n_group | E, 1 <= topk_group <= n_group <= 32,
    # k <= topk_group * E / n_group; the other routers ignore both fields
    (dict(router=2, n_group=4, topk_group=2), L.MOE_OK),
    (dict(router=2, E=256, k=8, n_group=8, topk_group=4), L.MOE_OK),
    (dict(router=2, E=256, k=8, n_group=32, topk_group=1), L.MOE_OK),
    (dict(router=2, n_group=1, topk_group=1), L.MOE_OK),
    (dict(router=2), L.MOE_ERR_INVALID_ARG),
    (dict(router=2, n_group=3, topk_group=1), L.MOE_ERR_INVALID_ARG),
    (dict(router=2, E=256, k=8, n_group=64, topk_group=8), L.MOE_ERR_INVALID_ARG),
    (dict(router=2, n_group=4, topk_group=0), L.MOE_ERR_INVALID_ARG),
    (dict(router=2, n_group=4, topk_group=5), L.MOE_ERR_INVALID_ARG),
    (dict(router=2, k=3, n_group=4, topk_group=1), L.MOE_ERR_INVALID_ARG),
    (dict(router=0, n_group=3, topk_group=7), L.MOE_OK),
    (dict(payload_fp8=3), L.MOE_ERR_INVALID_ARG),
    (dict(payload_fp8=2, payload_scale=0.04), L.MOE_OK),
    (dict(payload_fp8=2), L.MOE_ERR_INVALID_ARG),                       # scale 0
    (dict(payload_fp8=2, payload_scale=-1.0), L.MOE_ERR_INVALID_ARG),
    (dict(payload_fp8=2, payload_scale=float("inf")), L.MOE_ERR_INVALID_ARG),
    (dict(payload_fp8=2, payload_scale=float("nan")), L.MOE_ERR_INVALID_ARG),
    (dict(payload_fp8=2, payload_scale=0.04, dtype=0), L.MOE_ERR_UNSUPPORTED),
    (dict(payload_fp8=0, payload_scale=-5.0), L.MOE_OK),
    # the GEMM pair-tile width: the built-in choice (0) or forced to 256 / 512
    (dict(gemm_tile_n=256), L.MOE_OK),
    (dict(gemm_tile_n=512), L.MOE_OK),
    (dict(gemm_tile_n=128), L.MOE_ERR_INVALID_ARG),
    (dict(gemm_tile_n=-1), L.MOE_ERR_INVALID_ARG),
    # packed or gathered rows: gathering takes bf16 without FP8 payload or soft gating
    (dict(x_perm_mode=1), L.MOE_OK),
    (dict(x_perm_mode=2), L.MOE_OK),
    (dict(x_perm_mode=2, E=256, k=8), L.MOE_OK),
    (dict(x_perm_mode=3), L.MOE_ERR_INVALID_ARG),
    (dict(x_perm_mode=-1), L.MOE_ERR_INVALID_ARG),
    (dict(x_perm_mode=2, dtype=0), L.MOE_ERR_UNSUPPORTED),
    (dict(x_perm_mode=2, payload_fp8=1), L.MOE_ERR_UNSUPPORTED),
    (dict(x_perm_mode=2, router=3, E=8, k=8, tau=1.0), L.MOE_ERR_UNSUPPORTED),
    (dict(x_perm_mode=1, dtype=0), L.MOE_OK),
    (dict(output_fp8=1), L.MOE_OK),
    (dict(output_fp8=1, dtype=0), L.MOE_OK),
    (dict(output_fp8=2), L.MOE_ERR_INVALID_ARG),
    (dict(output_fp8=-1), L.MOE_ERR_INVALID_ARG),
    # soft gating: k = E <= 16, tau finite and > 0, no FP8 payload
    (dict(router=3, E=8, k=8, tau=1.0), L.MOE_OK),
    (dict(router=3, E=16, k=16, tau=0.5, output_fp8=1), L.MOE_OK),
    (dict(router=3, E=16, k=16, tau=0.5, dtype=0), L.MOE_OK),
    (dict(router=3, E=8, k=2, tau=1.0), L.MOE_ERR_INVALID_ARG),
    (dict(router=3, E=32, k=32, tau=1.0), L.MOE_ERR_INVALID_ARG),
    (dict(router=3, E=8, k=8, tau=0.0), L.MOE_ERR_INVALID_ARG),
    (dict(router=3, E=8, k=8, tau=float("nan")), L.MOE_ERR_INVALID_ARG),
    (dict(router=3, E=8, k=8, tau=1.0, payload_fp8=1), L.MOE_ERR_UNSUPPORTED),
    (dict(router=4), L.MOE_ERR_INVALID_ARG),
    (dict(payload_fp8=1, dtype=0), L.MOE_ERR_UNSUPPORTED),
    (dict(T=1 << 30, k=8), L.MOE_ERR_UNSUPPORTED),
    # the forward keeps Z for the backward: not with an FP8 payload
    (dict(keep_z=1), L.MOE_OK),
    (dict(keep_z=1, dtype=0), L.MOE_OK),
    (dict(keep_z=1, router=3, E=8, k=8, tau=1.0), L.MOE_OK),
    (dict(keep_z=1, x_perm_mode=2), L.MOE_OK),
    (dict(keep_z=2), L.MOE_ERR_INVALID_ARG),
    (dict(keep_z=-1), L.MOE_ERR_INVALID_ARG),
    (dict(keep_z=1, payload_fp8=1), L.MOE_ERR_UNSUPPORTED),
    (dict(keep_z=1, output_fp8=1), L.MOE_ERR_UNSUPPORTED),
])
def test_check_config(lib, kw, status):
    c = cfg(**kw)
    assert lib.moe_check_config(ctypes.byref(c)) == status
    if status != L.MOE_OK:
        assert lib.moe_workspace_size(ctypes.byref(c)) == 0
        assert lib.moe_scratch_size(ctypes.byref(c)) == 0
        assert lib.moe_forward_kernel_count(ctypes.byref(c)) == 0


def test_null_config(lib):
    assert lib.moe_check_config(None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_size(None) == 0


def test_workspace_sizes(lib):
    c = cfg(T=1024, d=4096, E=8, k=2, f=11008)
    ws = lib.moe_workspace_size(ctypes.byref(c))
    sc = lib.moe_scratch_size(ctypes.byref(c))
    R = 1024 * 2
    need = R * 4096 * 2 + R * 11008 * 2 + R * 4096 * 4   # x_perm + H + Y
    assert sc > 0 and ws >= sc + need
    assert ws < sc + need + (1 << 20)
    assert ws % 256 == 0 and sc % 256 == 0
    c8 = cfg(T=1024, d=4096, E=8, k=2, f=11008, payload_fp8=1)
    # the FP8 payload is expanded inside the W1 GEMM: no staging copy in
    # scratch and no kernel of its own; the forward workspace holds R*d
    # payload bytes (not 2*R*d) plus a scale per row
    assert lib.moe_scratch_size(ctypes.byref(c8)) == sc
    assert lib.moe_workspace_size(ctypes.byref(c8)) <= ws - R * 4096 + R * 4 + 256
    # R = T*k = 2048 <= 4096: dispatch is one kernel (each CTA counts all
    # ids); larger batches count, scan and scatter in three
    assert lib.moe_forward_kernel_count(ctypes.byref(c)) == 5
    assert lib.moe_forward_kernel_count(ctypes.byref(c8)) == 5
    cb = cfg(T=4096, d=4096, E=8, k=2, f=11008)
    assert lib.moe_forward_kernel_count(ctypes.byref(cb)) == 7
    # the FP8 expert-output payload: R*d bytes + scale and zero per row in
    # the forward workspace, one more kernel, no extra scratch
    co = cfg(T=1024, d=4096, E=8, k=2, f=11008, output_fp8=1)
    assert lib.moe_workspace_size(ctypes.byref(co)) >= ws + R * 4096 + R * 8
    assert lib.moe_scratch_size(ctypes.byref(co)) == sc
    assert lib.moe_forward_kernel_count(ctypes.byref(co)) == 6
    # soft gating packs no rows (the W1 GEMM reads x): the forward workspace
    # is R*d*2 bytes smaller than a top-k layer with the same fan-out; one
    # layout kernel instead of the three dispatch kernels
    cs = cfg(T=1024, d=4096, E=8, k=8, f=11008, router=3, tau=1.0)
    ck = cfg(T=1024, d=4096, E=8, k=8, f=11008)
    Rs = 1024 * 8
    assert lib.moe_workspace_size(ctypes.byref(ck)) - lib.moe_workspace_size(ctypes.byref(cs)) \
        >= Rs * 4096 * 2
    assert lib.moe_forward_kernel_count(ctypes.byref(cs)) == 5


@pytest.mark.parametrize("dtype", [0, 1])
def test_keep_z_workspaces(lib, dtype):
    # keep_z: the forward workspace holds Z (R*f fp32 more, aligned); a bf16
    # backward then reads it there and its own workspace drops the R*f fp32
    # of the recomputed Z, while an fp32 backward keeps it (dZ is formed in
    # place over a copy); the kernel count of the forward is unchanged
    c = cfg(T=1024, d=4096, E=8, k=2, f=11008, dtype=dtype)
    cz = cfg(T=1024, d=4096, E=8, k=2, f=11008, dtype=dtype, keep_z=1)
    R, f = 1024 * 2, 11008
    dws = lib.moe_workspace_size(ctypes.byref(cz)) - lib.moe_workspace_size(ctypes.byref(c))
    assert R * f * 4 <= dws <= R * f * 4 + 256
    assert lib.moe_scratch_size(ctypes.byref(cz)) == lib.moe_scratch_size(ctypes.byref(c))
    assert lib.moe_forward_kernel_count(ctypes.byref(cz)) == \
        lib.moe_forward_kernel_count(ctypes.byref(c))
    dbw = lib.moe_backward_workspace_size(ctypes.byref(c)) - \
        lib.moe_backward_workspace_size(ctypes.byref(cz))
    if dtype == 1:
        assert R * f * 4 <= dbw <= R * f * 4 + 256
    else:
        assert dbw == 0


def test_backward_workspace_follows_the_dw2_split_side(lib):
    # bf16 layers split dW2's fp32 operand on its narrower side: w H ([R][2f]
    # bf16) where 2f <= d, else dY ([R][2d]); growing d by 64 then changes the
    # backward workspace by the d-wide buffers only (dY's split when it is
    # the one kept, dX_perm, the dout rows, dx_gate), not by the split of w H
    T, E, k, f = 256, 8, 2, 128
    R = T * k
    def bws(d, dtype=1):
        c = cfg(T=T, d=d, E=E, k=k, f=f, dtype=dtype)
        return lib.moe_backward_workspace_size(ctypes.byref(c))
    # d-wide bytes per unit of d: dX_perm R*4, dout rows R*2, dx_gate T*4,
    # gate partials (token chunks * E * 4), and dY's split R*4 when kept
    d0, d1 = 256, 320                       # 2f = 256 <= d: w H split
    grow_h = bws(d1) - bws(d0)
    d2, d3 = 128, 192                       # 2f = 256 > d: dY split
    grow_y = bws(d3) - bws(d2)
    # the dY split adds R * 2 * 2 bytes per unit of d on the second pair only
    assert abs((grow_y - grow_h) - 64 * R * 4) <= 4 * 256
    # fp32 layers keep fp32 dY whichever is narrower
    assert bws(d1, 0) - bws(d0, 0) == bws(d3, 0) - bws(d2, 0)


FAKE = ctypes.c_void_p(0x100000)       # never dereferenced: validation fails first
FAKE_ODD = ctypes.c_void_p(0x100008)   # 8-byte aligned only


def test_forward_argument_errors(lib):
    c = cfg()
    n = lib.moe_workspace_size(ctypes.byref(c))
    f = lib.moe_forward
    assert f(None, FAKE, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, n, None) == L.MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(c), None, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, n, None) == L.MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(c), FAKE_ODD, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, n, None) == L.MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(c), FAKE, FAKE, None, None, FAKE, FAKE, FAKE, FAKE_ODD, n, None) == L.MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(c), FAKE, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, n - 1, None) == L.MOE_ERR_WORKSPACE_TOO_SMALL
    soft = cfg(router=3, E=8, k=8, tau=1.0)
    ns = lib.moe_workspace_size(ctypes.byref(soft))
    # the soft router needs its Gumbel samples
    assert f(ctypes.byref(soft), FAKE, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, ns, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_route(ctypes.byref(soft), FAKE, FAKE, None, None, FAKE, FAKE, None, None) == L.MOE_ERR_INVALID_ARG
    bad = cfg(d=96)
    assert f(ctypes.byref(bad), FAKE, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, n, None) == L.MOE_ERR_INVALID_ARG


def test_forward_with_events_wrong_count(lib):
    c = cfg()
    n = lib.moe_workspace_size(ctypes.byref(c))
    ev = (ctypes.c_void_p * 3)()
    assert lib.moe_forward_with_events(ctypes.byref(c), FAKE, FAKE, None, None, FAKE, FAKE, FAKE,
                                       FAKE, n, ev, 3, None) == L.MOE_ERR_INVALID_ARG


def test_stage_argument_errors(lib):
    c = cfg()
    sc = lib.moe_scratch_size(ctypes.byref(c))
    assert lib.moe_route(ctypes.byref(c), None, FAKE, None, None, FAKE, FAKE, None, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                            FAKE, sc - 1, None) == L.MOE_ERR_WORKSPACE_TOO_SMALL
    assert lib.moe_dispatch(ctypes.byref(c), FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                            FAKE, sc, None) == L.MOE_ERR_INVALID_ARG
    c8 = cfg(payload_fp8=1)
    sc8 = lib.moe_scratch_size(ctypes.byref(c8))
    assert lib.moe_dispatch(ctypes.byref(c8), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                            FAKE, sc8, None) == L.MOE_ERR_INVALID_ARG   # no x_scale
    assert lib.moe_expert_ffn(ctypes.byref(c), FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE_ODD,
                              FAKE, sc, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, None, sc, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_output(ctypes.byref(c), FAKE, FAKE_ODD, FAKE, FAKE, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_output(ctypes.byref(c), FAKE, FAKE, None, FAKE, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_combine_fp8(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, sc - 1,
                               None) == L.MOE_ERR_WORKSPACE_TOO_SMALL
    assert lib.moe_combine_fp8(ctypes.byref(c), FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, sc,
                               None) == L.MOE_ERR_INVALID_ARG
    # an empty batch needs no device work for routing
    c0 = cfg(T=0)
    assert lib.moe_route(ctypes.byref(c0), None, None, None, None, None, None, None, None) == L.MOE_OK


def test_backward_argument_errors(lib):
    c = cfg(T=1024, d=4096, E=8, k=2, f=11008)
    ws = lib.moe_workspace_size(ctypes.byref(c))
    bws = lib.moe_backward_workspace_size(ctypes.byref(c))
    R = 1024 * 2
    # per routed row: dY (fp32, or for bf16 layers its bf16 hi/lo split: the
    # same bytes), Z and dX_perm (fp32); and the gate part of dx
    assert bws >= R * 4096 * 4 * 2 + R * 11008 * 4 + 1024 * 4096 * 4
    args = lambda cc, fws, b: (ctypes.byref(cc), FAKE, FAKE, None, None, FAKE, FAKE, FAKE, fws,
                               FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, b, None)
    assert lib.moe_backward(*args(c, ws - 1, bws)) == L.MOE_ERR_WORKSPACE_TOO_SMALL
    assert lib.moe_backward(*args(c, ws, bws - 1)) == L.MOE_ERR_WORKSPACE_TOO_SMALL
    bad = list(args(c, ws, bws))
    bad[9] = None                                     # no dout
    assert lib.moe_backward(*bad) == L.MOE_ERR_INVALID_ARG
    bad = list(args(c, ws, bws))
    bad[7] = FAKE_ODD                                 # forward workspace misaligned
    assert lib.moe_backward(*bad) == L.MOE_ERR_INVALID_ARG
    for i in (9, 10, 13):                             # dout, dx, dW1 misaligned
        bad = list(args(c, ws, bws))
        bad[i] = FAKE_ODD
        assert lib.moe_backward(*bad) == L.MOE_ERR_INVALID_ARG
    # the FP8 payloads have no backward
    for c8 in (cfg(T=1024, d=4096, E=8, k=2, f=11008, payload_fp8=1),
               cfg(T=1024, d=4096, E=8, k=2, f=11008, output_fp8=1)):
        assert lib.moe_backward(*args(c8, 1 << 40, 1 << 40)) == L.MOE_ERR_UNSUPPORTED
    # soft gating needs the Gumbel samples
    cs = cfg(T=16, E=8, k=8, router=3, tau=1.0)
    assert lib.moe_backward(*args(cs, 1 << 40, 1 << 40)) == L.MOE_ERR_INVALID_ARG


def test_strerror(lib):
    for code in range(-6, 1):
        s = lib.moe_strerror(code).decode()
        assert s and s != "unknown status"
    assert lib.moe_strerror(-99).decode() == "unknown status"
    assert lib.moe_get_device_error(None, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_clear_device_error(None, None) == L.MOE_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(tmp_path):
    import importlib
    mod = importlib.import_module("mixture_experts_routed_gb300._lib")
    saved = mod._lib
    try:
        mod._lib = None
        with pytest.raises(RuntimeError, match="not built"):
            mod.load(str(tmp_path / "missing.so"))
    finally:
        mod._lib = saved


def test_binding_refuses_strided_and_host_tensors():
    # the Python binding hands the C ABI raw addresses: a transposed view or
    # a host tensor is refused before any call is made (no GPU needed)
    import torch
    import mixture_experts_routed_gb300 as moe
    from workloads import get_config
    c = get_config("tiny_T256_d128_E8_k2_f256_fp32")
    Wg = torch.zeros((c.d, c.E))
    with pytest.raises(moe.MoEError, match="not contiguous"):
        moe.route(c, torch.zeros((c.d, c.T)).t(), Wg)
    with pytest.raises(moe.MoEError, match="not in GPU memory"):
        moe.route(c, torch.zeros((c.T, c.d)), Wg)


@pytest.mark.parametrize("compiler,std", [("gcc", "-std=c11"), ("g++", "-std=c++17")])
def test_header_compiles_as_plain_c_and_cpp(tmp_path, compiler, std):
    # a C ABI: the header alone, warnings as errors, in C and in C++
    if subprocess.run(["which", compiler], capture_output=True).returncode != 0:
        pytest.skip(f"{compiler} not installed")
    src = tmp_path / "use_moe.c"
    src.write_text('#include "moe.h"\n'
                   "int use(const moe_config_t* c) { return moe_check_config(c); }\n")
    lang = ["-x", "c++"] if compiler == "g++" else []
    r = subprocess.run([compiler, std, "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-fsyntax-only", *lang, "-I", os.path.join(ROOT, "include"), str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
