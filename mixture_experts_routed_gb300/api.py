"""Python binding of the routed-MoE layer library: the same entry points as
include/moe.h, taking torch tensors.

Marshalling only: every step of the layer runs in the CUDA library. torch is
used for device memory (outputs a caller does not pass are allocated with
torch), for the current stream, and nothing else. There is no fallback: if
the library is missing, importing the first call raises.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib as L

__all__ = ["MoEError", "make_config", "config_from", "workspace_size", "scratch_size",
           "alloc_workspace", "route", "dispatch", "expert_ffn", "combine", "forward",
           "forward_views", "get_device_error", "clear_device_error", "kernel_count",
           "check_config", "backward", "backward_workspace_size"]


class MoEError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = L.load().moe_strerror(status).decode()
        super().__init__(f"{what}: {msg} (status {status})" if what else msg)


def make_config(T, d, E, k, f, dtype="bf16", router=L.MOE_ROUTER_RENORM, pre_k=8,
                payload_fp8=0, n_group=1, topk_group=1, payload_scale=0.0,
                output_fp8=0, tau=1.0, gemm_tile_n=0, x_perm_mode=0, keep_z=0) -> L.MoeConfig:
    dt = {"f32": L.MOE_DTYPE_F32, "fp32": L.MOE_DTYPE_F32, "bf16": L.MOE_DTYPE_BF16,
          torch.float32: L.MOE_DTYPE_F32, torch.bfloat16: L.MOE_DTYPE_BF16}[dtype]
    return L.MoeConfig(int(T), int(d), int(E), int(k), int(f), dt, int(router), int(pre_k),
                       int(payload_fp8), int(n_group), int(topk_group), float(payload_scale),
                       int(output_fp8), float(tau), int(gemm_tile_n), int(x_perm_mode),
                       int(keep_z))


def config_from(c) -> L.MoeConfig:
    """From any object with T, d, E, k, f, dtype, router, pre_k, payload_fp8
    (and, optionally, n_group, topk_group, payload_scale, output_fp8, tau,
    gemm_tile_n, x_perm_mode, keep_z)."""
    if isinstance(c, L.MoeConfig):
        return c
    return make_config(c.T, c.d, c.E, c.k, c.f, c.dtype, c.router, c.pre_k, c.payload_fp8,
                       getattr(c, "n_group", 1), getattr(c, "topk_group", 1),
                       getattr(c, "payload_scale", 0.0), getattr(c, "output_fp8", 0),
                       getattr(c, "tau", 1.0), getattr(c, "gemm_tile_n", 0),
                       getattr(c, "x_perm_mode", 0), getattr(c, "keep_z", 0))


def _cfg(c):
    return ctypes.byref(config_from(c))


def _p(t):
    """Device address of a dense CUDA tensor: the C ABI takes row-major
    buffers in GPU memory, so a strided view (read with the wrong layout) or
    a host tensor (an address no kernel may touch) is refused here."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise MoEError(L.MOE_ERR_INVALID_ARG, "tensor is not contiguous")
    if not t.is_cuda:
        raise MoEError(L.MOE_ERR_INVALID_ARG, "tensor is not in GPU memory")
    return ctypes.c_void_p(t.data_ptr())


def _s(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(st, what):
    if st != L.MOE_OK:
        raise MoEError(st, what)


def _dt(c):
    return torch.float32 if config_from(c).dtype == L.MOE_DTYPE_F32 else torch.bfloat16


def check_config(c) -> int:
    return L.load().moe_check_config(_cfg(c))


def workspace_size(c) -> int:
    return L.load().moe_workspace_size(_cfg(c))


def scratch_size(c) -> int:
    return L.load().moe_scratch_size(_cfg(c))


def kernel_count(c) -> int:
    return L.load().moe_forward_kernel_count(_cfg(c))


def backward_workspace_size(c) -> int:
    return int(L.load().moe_backward_workspace_size(_cfg(c)))


def alloc_workspace(c, kind: str = "forward", device=None) -> torch.Tensor:
    """Zeroed workspace (so the device error word starts clear); kind is
    "forward", "scratch" or "backward"."""
    n = {"forward": workspace_size, "scratch": scratch_size,
         "backward": backward_workspace_size}[kind](c)
    if n == 0:
        raise MoEError(L.MOE_ERR_INVALID_ARG, "workspace size")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def route(c, x, Wg, bias=None, *, noise=None, topk_idx=None, topk_w=None, logits=None,
          want_logits=False, stream=None):
    """Gate + router. ``noise``: the soft router's Gumbel samples [T, E]."""
    cc = config_from(c)
    dev = x.device
    if topk_idx is None:
        topk_idx = torch.empty((cc.T, cc.k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((cc.T, cc.k), dtype=torch.float32, device=dev)
    if logits is None and want_logits:
        logits = torch.empty((cc.T, cc.E), dtype=torch.float32, device=dev)
    st = L.load().moe_route(ctypes.byref(cc), _p(x), _p(Wg), _p(bias), _p(noise),
                            _p(topk_idx), _p(topk_w), _p(logits), _s(stream))
    _check(st, "moe_route")
    return topk_idx, topk_w, logits


def dispatch(c, x, topk_idx, *, ws, counts=None, offsets=None, pos=None, src=None,
             x_perm=None, x_scale=None, stream=None) -> dict:
    cc = config_from(c)
    dev = x.device
    R = cc.T * cc.k
    i32 = dict(dtype=torch.int32, device=dev)
    counts = torch.empty(cc.E, **i32) if counts is None else counts
    offsets = torch.empty(cc.E + 1, **i32) if offsets is None else offsets
    pos = torch.empty(R, **i32) if pos is None else pos
    src = torch.empty(R, **i32) if src is None else src
    soft = cc.router == L.MOE_ROUTER_SOFT_GUMBEL
    if x_perm is None and not soft:       # soft gating packs no rows
        pdt = torch.uint8 if cc.payload_fp8 else _dt(cc)
        x_perm = torch.empty((R, cc.d), dtype=pdt, device=dev)
    if x_scale is None and cc.payload_fp8:
        x_scale = torch.empty(R, dtype=torch.float32, device=dev)
    st = L.load().moe_dispatch(ctypes.byref(cc), _p(x), _p(topk_idx), _p(counts), _p(offsets),
                               _p(pos), _p(src), _p(x_perm), _p(x_scale), _p(ws),
                               ws.numel() * ws.element_size(), _s(stream))
    _check(st, "moe_dispatch")
    return {"counts": counts, "offsets": offsets, "pos": pos, "src": src, "x_perm": x_perm,
            "x_scale": x_scale}


def expert_ffn(c, x_perm, x_scale, offsets, W1, W2, *, ws, h=None, y_perm=None, stream=None):
    """Grouped FFN. With the soft router ``x_perm`` is x itself ([T, d])."""
    cc = config_from(c)
    dev = x_perm.device
    R = cc.T * cc.k
    if h is None:
        h = torch.empty((R, cc.f), dtype=_dt(cc), device=dev)
    if y_perm is None:
        y_perm = torch.empty((R, cc.d), dtype=torch.float32, device=dev)
    st = L.load().moe_expert_ffn(ctypes.byref(cc), _p(x_perm), _p(x_scale), _p(offsets),
                                 _p(W1), _p(W2), _p(h), _p(y_perm), _p(ws),
                                 ws.numel() * ws.element_size(), _s(stream))
    _check(st, "moe_expert_ffn")
    return h, y_perm


def combine(c, y_perm, pos, topk_w, *, ws, out=None, stream=None):
    cc = config_from(c)
    if out is None:
        out = torch.empty((cc.T, cc.d), dtype=_dt(cc), device=y_perm.device)
    st = L.load().moe_combine(ctypes.byref(cc), _p(y_perm), _p(pos), _p(topk_w), _p(out),
                              _p(ws), ws.numel() * ws.element_size(), _s(stream))
    _check(st, "moe_combine")
    return out


def quantize_output(c, y_perm, *, y_q=None, y_scale=None, y_zero=None, stream=None):
    """FP8 expert-output payload: (y_q uint8 [R, d], y_scale [R], y_zero [R])."""
    cc = config_from(c)
    R, dev = cc.T * cc.k, y_perm.device
    if y_q is None:
        y_q = torch.empty((R, cc.d), dtype=torch.uint8, device=dev)
    if y_scale is None:
        y_scale = torch.empty((R,), dtype=torch.float32, device=dev)
    if y_zero is None:
        y_zero = torch.empty((R,), dtype=torch.float32, device=dev)
    st = L.load().moe_quantize_output(ctypes.byref(cc), _p(y_perm), _p(y_q), _p(y_scale),
                                      _p(y_zero), _s(stream))
    _check(st, "moe_quantize_output")
    return y_q, y_scale, y_zero


def combine_fp8(c, y_q, y_scale, y_zero, pos, topk_w, *, ws, out=None, stream=None):
    cc = config_from(c)
    if out is None:
        out = torch.empty((cc.T, cc.d), dtype=_dt(cc), device=y_q.device)
    st = L.load().moe_combine_fp8(ctypes.byref(cc), _p(y_q), _p(y_scale), _p(y_zero), _p(pos),
                                  _p(topk_w), _p(out), _p(ws), ws.numel() * ws.element_size(),
                                  _s(stream))
    _check(st, "moe_combine_fp8")
    return out


def forward(c, x, Wg, bias, W1, W2, *, ws, out=None, events=None, noise=None, stream=None):
    """The whole layer. ``events``: optional list of MOE_NUM_EVENTS
    torch.cuda.Event (or None) recorded at the kernel boundaries. ``noise``:
    the soft router's Gumbel samples [T, E]."""
    cc = config_from(c)
    if out is None:
        out = torch.empty((cc.T, cc.d), dtype=_dt(cc), device=x.device)
    lib = L.load()
    nbytes = ws.numel() * ws.element_size()
    if events is None:
        st = lib.moe_forward(ctypes.byref(cc), _p(x), _p(Wg), _p(bias), _p(noise), _p(W1),
                             _p(W2), _p(out), _p(ws), nbytes, _s(stream))
    else:
        strm = stream if stream is not None else torch.cuda.current_stream()
        for e in events:
            if e is not None and not e.cuda_event:
                e.record(strm)          # torch creates its CUDA event lazily
        arr = (ctypes.c_void_p * L.MOE_NUM_EVENTS)(
            *[None if e is None else e.cuda_event for e in events])
        st = lib.moe_forward_with_events(ctypes.byref(cc), _p(x), _p(Wg), _p(bias), _p(noise),
                                         _p(W1), _p(W2), _p(out), _p(ws), nbytes, arr,
                                         len(events), _s(stream))
    _check(st, "moe_forward")
    return out


def backward(c, x, Wg, bias, W1, W2, dout, *, fwd_ws, ws, noise=None, stream=None) -> dict:
    """Gradients of the layer for dout = dl/dout [T, d] after a forward in
    ``fwd_ws`` on the same inputs: dx [T, d], dWg [d, E], dbias [E], dW1 [E,
    d, f], dW2 [E, f, d], all fp32. ``ws``: a backward workspace."""
    cc = config_from(c)
    dev = x.device
    g = {"dx": torch.empty((cc.T, cc.d), dtype=torch.float32, device=dev),
         "dWg": torch.empty((cc.d, cc.E), dtype=torch.float32, device=dev),
         "dbias": torch.empty((cc.E,), dtype=torch.float32, device=dev),
         "dW1": torch.empty((cc.E, cc.d, cc.f), dtype=torch.float32, device=dev),
         "dW2": torch.empty((cc.E, cc.f, cc.d), dtype=torch.float32, device=dev)}
    st = L.load().moe_backward(
        ctypes.byref(cc), _p(x), _p(Wg), _p(bias), _p(noise), _p(W1), _p(W2), _p(fwd_ws),
        fwd_ws.numel() * fwd_ws.element_size(), _p(dout), _p(g["dx"]), _p(g["dWg"]),
        _p(g["dbias"]), _p(g["dW1"]), _p(g["dW2"]), _p(ws), ws.numel() * ws.element_size(),
        _s(stream))
    _check(st, "moe_backward")
    return g


def forward_views(c, ws) -> dict:
    """Tensors viewing the intermediates of the last forward in ``ws``."""
    cc = config_from(c)
    v = L.MoeForwardViews()
    _check(L.load().moe_forward_views(ctypes.byref(cc), _p(ws), ctypes.byref(v)),
           "moe_forward_views")
    base = ws.data_ptr()
    R = cc.T * cc.k

    def view(ptr, n, dtype, shape):
        if ptr is None:
            return None
        off = ptr - base
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return ws[off:off + nbytes].view(dtype).view(shape)

    pdt = torch.uint8 if cc.payload_fp8 else _dt(cc)
    return {
        "topk_idx": view(v.topk_idx, R, torch.int32, (cc.T, cc.k)),
        "topk_w": view(v.topk_w, R, torch.float32, (cc.T, cc.k)),
        "counts": view(v.counts, cc.E, torch.int32, (cc.E,)),
        "offsets": view(v.offsets, cc.E + 1, torch.int32, (cc.E + 1,)),
        "pos": view(v.pos, R, torch.int32, (R,)),
        "src": view(v.src, R, torch.int32, (R,)),
        "x_perm": view(v.x_perm, R * cc.d, pdt, (R, cc.d)) if v.x_perm else None,
        "x_scale": view(v.x_scale, R, torch.float32, (R,)) if cc.payload_fp8 else None,
        "h": view(v.h, R * cc.f, _dt(cc), (R, cc.f)),
        "y_perm": view(v.y_perm, R * cc.d, torch.float32, (R, cc.d)),
        "y_q": view(v.y_q, R * cc.d, torch.uint8, (R, cc.d)) if cc.output_fp8 else None,
        "y_scale": view(v.y_scale, R, torch.float32, (R,)) if cc.output_fp8 else None,
        "y_zero": view(v.y_zero, R, torch.float32, (R,)) if cc.output_fp8 else None,
        "z": view(v.z, R * cc.f, torch.float32, (R, cc.f)) if cc.keep_z else None,
    }


def get_device_error(ws, stream=None) -> int:
    """Synchronise, read and clear the workspace error word (a moe status)."""
    return L.load().moe_get_device_error(_p(ws), _s(stream))


def clear_device_error(ws, stream=None) -> None:
    _check(L.load().moe_clear_device_error(_p(ws), _s(stream)), "moe_clear_device_error")
