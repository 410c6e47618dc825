"""ctypes declarations of the C ABI in include/moe.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_WORKSPACE_TOO_SMALL = -3
MOE_ERR_LAUNCH = -4
MOE_ERR_BAD_INDEX = -5
MOE_ERR_TIMEOUT = -6

MOE_DTYPE_F32 = 0
MOE_DTYPE_BF16 = 1
MOE_ROUTER_RENORM = 0
MOE_ROUTER_PREK_SOFTMAX = 1
MOE_ROUTER_GROUP_LIMITED = 2
MOE_ROUTER_SOFT_GUMBEL = 3
MOE_NUM_EVENTS = 8
MOE_XPERM_AUTO = 0
MOE_XPERM_PACKED = 1
MOE_XPERM_GATHERED = 2


class MoeConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("T", "d", "E", "k", "f", "dtype", "router", "pre_k", "payload_fp8",
                 "n_group", "topk_group")] + [("payload_scale", ctypes.c_float),
                                             ("output_fp8", ctypes.c_int32),
                                             ("tau", ctypes.c_float),
                                             ("gemm_tile_n", ctypes.c_int32),
                                             ("x_perm_mode", ctypes.c_int32),
                                             ("keep_z", ctypes.c_int32)]


class MoeForwardViews(ctypes.Structure):
    _fields_ = [("topk_idx", ctypes.c_void_p), ("topk_w", ctypes.c_void_p),
                ("counts", ctypes.c_void_p), ("offsets", ctypes.c_void_p),
                ("pos", ctypes.c_void_p), ("src", ctypes.c_void_p),
                ("x_perm", ctypes.c_void_p), ("x_scale", ctypes.c_void_p),
                ("h", ctypes.c_void_p), ("y_perm", ctypes.c_void_p),
                ("y_q", ctypes.c_void_p), ("y_scale", ctypes.c_void_p),
                ("y_zero", ctypes.c_void_p), ("z", ctypes.c_void_p)]


_P = ctypes.c_void_p
_CFG = ctypes.POINTER(MoeConfig)
_SZ = ctypes.c_size_t
_I = ctypes.c_int

# name -> (restype, argtypes); the same names as include/moe.h
PROTOTYPES = {
    "moe_check_config": (_I, [_CFG]),
    "moe_scratch_size": (_SZ, [_CFG]),
    "moe_workspace_size": (_SZ, [_CFG]),
    "moe_route": (_I, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_dispatch": (_I, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_expert_ffn": (_I, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_combine": (_I, [_CFG, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_quantize_output": (_I, [_CFG, _P, _P, _P, _P, _P]),
    "moe_combine_fp8": (_I, [_CFG, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward": (_I, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_with_events": (_I, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                     ctypes.POINTER(ctypes.c_void_p), _I, _P]),
    "moe_forward_views": (_I, [_CFG, _P, ctypes.POINTER(MoeForwardViews)]),
    "moe_get_device_error": (_I, [_P, _P]),
    "moe_clear_device_error": (_I, [_P, _P]),
    "moe_strerror": (ctypes.c_char_p, [_I]),
    "moe_forward_kernel_count": (_I, [_CFG]),
    "moe_set_gemm_epilogue_wait_ns": (_I, [ctypes.c_uint64]),
    "moe_dispatch_noalloc": (_I, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_backward_workspace_size": (_SZ, [_CFG]),
    "moe_backward": (_I, [_CFG, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P, _P, _P, _P, _P, _P,
                          _SZ, _P]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library. Raises if it has not been built: there is no
    fallback implementation."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{os.path.basename(path)} is not built: run "
            "`python -m mixture_experts_routed_gb300.build` (needs nvcc, sm_103a)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in PROTOTYPES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
