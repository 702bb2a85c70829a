"""GB300-native routed-expert MoE hot path: permute, grouped matmul (tcgen05),
clipped SwiGLU, weighted combine, and their gradients, behind the C ABI in
include/moe_gmm.h; the MX (MXFP8 / MXFP4) forward behind include/moe_mx.h.  This
package is the Python binding of that library; all computation runs in its CUDA
kernels (there is no fallback)."""
from .binding import (  # noqa: F401
    LayerSaved, MoeError, Workspace, gmm_backward, gmm_backward_dx_swiglu, gmm_forward, gmm_workspace_size, moe_layer_backward,
    moe_layer_forward, moe_layer_workspace_size, moe_permute, moe_permute_backward, moe_permute_no_alloc, moe_permute_workspace_size,
    moe_swiglu_backward, moe_unpermute, moe_unpermute_backward, moe_unpermute_workspace_size, read_status,
    status_string, moe_mx_quantize, moe_permute_mx, gmm_forward_mx, moe_layer_forward_mx, moe_layer_mx_workspace_size,
    check_wait_timeout, check_bounds, activation_format, gmm_forward_gather_act, gmm_forward_combine,
    gmm_forward_combine_workspace_size, moe_expert_mlp_forward, moe_expert_mlp_workspace_size,
)
from ._abi import MOE_EPILOGUE_NONE, MOE_EPILOGUE_SWIGLU, STATUS_NAMES, bounds_checking, load, lib_path  # noqa: F401
