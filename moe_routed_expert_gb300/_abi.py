"""ctypes view of the C ABI declared in include/moe_gmm.h and include/moe_mx.h (signatures only)."""
from __future__ import annotations

import ctypes as C
import os

from . import build as _build

P = C.c_void_p
I64 = C.c_int64
SZ = C.c_size_t
F32 = C.c_float
INT = C.c_int
ST = C.c_int  # moe_status_t

MOE_STATUS_BYTES = 256
MOE_EPILOGUE_NONE = 0
MOE_EPILOGUE_SWIGLU = 1

STATUS_NAMES = {
    0: "MOE_OK", 1: "MOE_ERR_NULLPTR", 2: "MOE_ERR_INVALID", 3: "MOE_ERR_UNSUPPORTED",
    4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE", 6: "MOE_ERR_TIMEOUT", 7: "MOE_ERR_BOUNDS",
}


FP8_FORMATS = {"e4m3": 0, "e5m2": 1, "e2m1": 5}  # moe_fp8_format_t (e2m1: packed two per byte)

ACTIVATIONS = {"swiglu": 0, "swiglustep": 1, "swigluoai": 2, "situglu": 3}  # moe_act_kind_t


class MoeActivation(C.Structure):
    _fields_ = [("kind", C.c_int32), ("n_params", C.c_int32), ("params", C.c_float * 3)]


class MoeLayerSaved(C.Structure):
    _fields_ = [("x_perm", P), ("h", P), ("a", P), ("y2", P),
                ("row_id_map", P), ("sorted_flat", P), ("group_list", P)]


SIGNATURES = {
    "moe_workspace_init": (ST, [P, SZ, P]),
    "moe_read_status": (ST, [P, P]),
    "moe_status_string": (C.c_char_p, [ST]),
    "moe_check_wait_timeout": (ST, [P, SZ, C.c_uint64, P]),
    "moe_check_bounds": (ST, [P, SZ, P]),
    "moe_permute_workspace_size": (SZ, [I64, I64, I64]),
    "moe_permute": (ST, [P, P, I64, I64, I64, I64, P, P, P, P, P, SZ, P]),
    "moe_permute_no_alloc": (ST, [P, P, I64, I64, I64, I64, P, P, P, P, P, P]),
    "gmm_workspace_size": (SZ, [I64, I64, I64, I64]),
    "gmm_forward": (ST, [P, P, P, I64, I64, I64, I64, INT, F32, P, P, P, SZ, P]),
    "gmm_backward": (ST, [P, P, P, P, I64, I64, I64, I64, P, P, P, SZ, P]),
    "gmm_backward_ex": (ST, [P, P, P, P, I64, I64, I64, I64, INT, P, P, P, SZ, P]),
    "gmm_forward_act": (ST, [P, P, P, I64, I64, I64, I64, C.POINTER(MoeActivation), INT, P, P, P, SZ, P]),
    "gmm_forward_gather_act": (ST, [P, P, I64, I64, P, P, I64, I64, I64, I64, C.POINTER(MoeActivation), INT, P,
                                    P, SZ, P]),
    "gmm_forward_combine_workspace_size": (SZ, [I64, I64, I64, I64]),
    "moe_expert_mlp_workspace_size": (SZ, [I64, I64, I64]),
    "moe_expert_mlp_forward": (ST, [P, P, P, P, P, I64, I64, I64, I64, I64, C.POINTER(MoeActivation), P, P, P, SZ,
                                    P]),
    "gmm_forward_combine": (ST, [P, P, P, P, P, P, I64, I64, I64, I64, I64, I64, INT, P, P, SZ, P]),
    "gmm_backward_dx_swiglu": (ST, [P, P, P, P, I64, I64, I64, I64, F32, P, P, SZ, P]),
    "gmm_backward_dx_act": (ST, [P, P, P, P, I64, I64, I64, I64, C.POINTER(MoeActivation), INT, P, P, SZ, P]),
    "moe_unpermute_workspace_size": (SZ, []),
    "moe_unpermute": (ST, [P, P, P, I64, I64, I64, P, P, SZ, P]),
    "moe_unpermute_backward": (ST, [P, P, P, P, I64, I64, I64, P, P, P, SZ, P]),
    "moe_permute_backward": (ST, [P, P, I64, I64, I64, P, P, SZ, P]),
    "moe_swiglu_backward": (ST, [P, P, I64, I64, F32, P, P, SZ, P]),
    "moe_activation_backward": (ST, [P, P, I64, I64, C.POINTER(MoeActivation), P, P, SZ, P]),
    "moe_layer_workspace_size": (SZ, [I64, I64, I64, I64, I64]),
    "moe_layer_forward": (ST, [P, P, P, P, P, I64, I64, I64, I64, I64, F32, P, C.POINTER(MoeLayerSaved),
                               P, SZ, P]),
    "moe_layer_backward": (ST, [P, P, P, P, C.POINTER(MoeLayerSaved), I64, I64, I64, I64, I64, F32,
                                P, P, P, P, P, SZ, P]),
    "moe_layer_forward_act": (ST, [P, P, P, P, P, I64, I64, I64, I64, I64, C.POINTER(MoeActivation), INT, P,
                                   C.POINTER(MoeLayerSaved), P, SZ, P]),
    "moe_layer_backward_act": (ST, [P, P, P, P, C.POINTER(MoeLayerSaved), I64, I64, I64, I64, I64,
                                    C.POINTER(MoeActivation), INT, P, P, P, P, P, SZ, P]),
    # moe_mx.h
    "moe_mx_quantize_workspace_size": (SZ, []),
    "moe_mx_quantize": (ST, [P, I64, I64, C.c_int32, P, P, P, SZ, P]),
    "moe_permute_mx": (ST, [P, P, I64, I64, I64, I64, C.c_int32, P, P, P, P, P, P, SZ, P]),
    "gmm_mx_workspace_size": (SZ, [I64, I64, I64, I64]),
    "gmm_forward_mx": (ST, [P, P, P, P, P, I64, I64, I64, I64, C.c_int32, C.c_int32, C.POINTER(MoeActivation),
                            P, P, P, P, P, SZ, P]),
    "moe_layer_mx_workspace_size": (SZ, [I64, I64, I64, I64, I64]),
    "moe_layer_forward_mx": (ST, [P, P, P, P, P, P, P, I64, I64, I64, I64, I64, C.c_int32, C.c_int32,
                                  C.POINTER(MoeActivation), P, P, SZ, P]),
}

_lib = None


def bounds_checking() -> bool:
    """MOE_GB300_BOUNDS_CHECK=1 selects the bounds-checking build of the library."""
    return os.environ.get("MOE_GB300_BOUNDS_CHECK", "") == "1"


def lib_path() -> str:
    return _build.BOUNDS_LIB_PATH if bounds_checking() else _build.LIB_PATH


def load(build_if_missing: bool = False):
    """Load the CUDA library (raises if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError("moe_routed_expert_gb300: CUDA library not built (%s); run build()" % path)
        _build.build(bounds=bounds_checking())
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
