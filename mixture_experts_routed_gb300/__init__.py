"""GB300-native routed mixture-of-experts layer (forward and backward).

The layer (gate -> softmax/top-k router -> dispatch -> grouped expert FFN ->
combine) runs as hand-written sm_103a CUDA kernels behind the C ABI in
include/moe.h; this package is its thin Python binding (``api``), the in-tree
build (``build``) and host-side load statistics (``stats``).
"""
from . import _lib  # noqa: F401
from .api import (  # noqa: F401
    MoEError, make_config, config_from, workspace_size, scratch_size, alloc_workspace, route,
    dispatch, expert_ffn, combine, quantize_output, combine_fp8, forward, forward_views,
    get_device_error,
    clear_device_error, kernel_count, check_config, backward, backward_workspace_size,
)
from ._lib import (  # noqa: F401
    MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE_TOO_SMALL,
    MOE_ERR_LAUNCH, MOE_ERR_BAD_INDEX, MOE_ERR_TIMEOUT, MOE_DTYPE_F32, MOE_DTYPE_BF16,
    MOE_ROUTER_RENORM, MOE_ROUTER_PREK_SOFTMAX, MOE_ROUTER_GROUP_LIMITED,
    MOE_ROUTER_SOFT_GUMBEL, MOE_NUM_EVENTS, MOE_XPERM_AUTO, MOE_XPERM_PACKED, MOE_XPERM_GATHERED,
)
