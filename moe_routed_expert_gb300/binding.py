"""Python binding of the C ABI: same names as include/moe_gmm.h, torch tensors in
and out.  Argument marshalling only -- every step runs in the CUDA library;
there is no CPU or PyTorch fallback, and a missing library raises.

Tensors must be CUDA, contiguous, and of the dtypes the header states (bf16
for activations and weights, int32 ids / row maps, int64 group_list, fp32
routing weights and dprobs).  Outputs are allocated here with torch (device
memory is torch's job) unless passed in.  Calls run on torch's current
stream unless ``stream`` is given.  Each call checks the host-side status;
device-side errors are sticky in the workspace and are read by
``read_status`` (which synchronises).
"""
from __future__ import annotations

import ctypes as C
from typing import Optional

import torch

from . import _abi

BF16 = torch.bfloat16


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s" % (where, _abi.STATUS_NAMES.get(status, str(status))))


def _lib():
    return _abi.load()


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status: int, where: str):
    if status != 0:
        raise MoeError(status, where)


def _dtype(t, dt, name):
    if t is not None and t.dtype != dt:
        raise ValueError("%s must be %s, got %s" % (name, dt, t.dtype))


class Workspace:
    """Caller-owned device workspace: zero-initialised status block + scratch."""

    def __init__(self, nbytes: int, device=None):
        self.nbytes = int(max(nbytes, _abi.MOE_STATUS_BYTES))
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device or "cuda")

    def ensure(self, nbytes: int) -> "Workspace":
        if nbytes > self.nbytes:
            self.__init__(nbytes, self.buf.device)
        return self

    @property
    def ptr(self):
        return C.c_void_p(self.buf.data_ptr())

    def reset(self, stream=None):
        _check(_lib().moe_workspace_init(self.ptr, self.nbytes, _stream(stream)), "moe_workspace_init")


def _ws(ws: Optional[Workspace], nbytes: int, device) -> Workspace:
    return Workspace(nbytes, device) if ws is None else ws.ensure(nbytes)


def read_status(ws: Workspace, stream=None) -> int:
    """Synchronise and return the workspace's sticky device status (0 = OK)."""
    return int(_lib().moe_read_status(ws.ptr, _stream(stream)))


def status_string(status: int) -> str:
    return _lib().moe_status_string(status).decode()


def check_bounds(ws: Workspace, stream=None):
    """Run the library's bounds-check self-check (see moe_check_bounds): afterwards
    read_status(ws) is MOE_ERR_BOUNDS (7) on the bounds-checking build, MOE_OK on
    the release build."""
    _check(_lib().moe_check_bounds(ws.ptr, ws.nbytes, _stream(stream)), "moe_check_bounds")


def check_wait_timeout(ws: Workspace, timeout_ns: int = 1000000, stream=None):
    """Run the library's bounded-wait failure check (see moe_check_wait_timeout):
    afterwards read_status(ws) is MOE_ERR_TIMEOUT (6)."""
    _check(_lib().moe_check_wait_timeout(ws.ptr, ws.nbytes, int(timeout_ns), _stream(stream)),
           "moe_check_wait_timeout")


# ------------------------------------------------------------------ sizes
def moe_permute_workspace_size(T, k, E) -> int:
    return int(_lib().moe_permute_workspace_size(T, k, E))


def gmm_workspace_size(M, K, N, E) -> int:
    return int(_lib().gmm_workspace_size(M, K, N, E))


def moe_unpermute_workspace_size() -> int:
    return int(_lib().moe_unpermute_workspace_size())


def moe_layer_workspace_size(T, H, I, E, k) -> int:
    return int(_lib().moe_layer_workspace_size(T, H, I, E, k))


# ------------------------------------------------------------------ dispatch
def moe_permute(x: Optional[torch.Tensor], topk_ids: torch.Tensor, E: int, *, out=None,
                ws: Optional[Workspace] = None, stream=None):
    """Returns (x_perm [T*k, H] or None, group_list [E] int64, row_id_map [T*k] int32,
    sorted_flat [T*k] int32)."""
    _dtype(x, BF16, "x")
    _dtype(topk_ids, torch.int32, "topk_ids")
    T, k = topk_ids.shape
    H = x.shape[1] if x is not None else 0
    dev = topk_ids.device
    if out is None:
        x_perm = torch.empty(T * k, H, dtype=BF16, device=dev) if x is not None else None
        group_list = torch.empty(E, dtype=torch.int64, device=dev)
        row_id_map = torch.empty(T * k, dtype=torch.int32, device=dev)
        sorted_flat = torch.empty(T * k, dtype=torch.int32, device=dev)
    else:
        x_perm, group_list, row_id_map, sorted_flat = out
    w = _ws(ws, moe_permute_workspace_size(T, k, E), dev)
    _check(_lib().moe_permute(_ptr(x), _ptr(topk_ids), T, H, k, E, _ptr(x_perm), _ptr(group_list),
                              _ptr(row_id_map), _ptr(sorted_flat), w.ptr, w.nbytes, _stream(stream)),
           "moe_permute")
    return x_perm, group_list, row_id_map, sorted_flat


def moe_permute_no_alloc(x: Optional[torch.Tensor], topk_ids: torch.Tensor, E: int, *, out=None,
                         device_status: Optional[torch.Tensor] = None, stream=None):
    """moe_permute without a workspace, for callers that cannot allocate device
    memory (the library's fixed internal scratch is used instead; see the C
    header for its size limit and for the rule that overlapping calls race).
    Outputs are allocated here only when ``out`` is not given."""
    _dtype(x, BF16, "x")
    _dtype(topk_ids, torch.int32, "topk_ids")
    T, k = topk_ids.shape
    H = x.shape[1] if x is not None else 0
    dev = topk_ids.device
    if out is None:
        out = (torch.empty(T * k, H, dtype=BF16, device=dev) if x is not None else None,
               torch.empty(E, dtype=torch.int64, device=dev),
               torch.empty(T * k, dtype=torch.int32, device=dev),
               torch.empty(T * k, dtype=torch.int32, device=dev))
    x_perm, group_list, row_id_map, sorted_flat = out
    _check(_lib().moe_permute_no_alloc(_ptr(x), _ptr(topk_ids), T, H, k, E, _ptr(x_perm), _ptr(group_list),
                                       _ptr(row_id_map), _ptr(sorted_flat), _ptr(device_status), _stream(stream)),
           "moe_permute_no_alloc")
    return x_perm, group_list, row_id_map, sorted_flat


# ------------------------------------------------------------------ gated activations
def _act(activation):
    """(kind, params) -> the C moe_activation_t: kind one of "swiglu",
    "swiglustep", "swigluoai", "situglu"; params the activation_params list
    (its defaults and checks are the library's)."""
    kind, params = activation if isinstance(activation, tuple) else (activation, ())
    if kind not in _abi.ACTIVATIONS:
        raise ValueError("unknown activation %r" % (kind,))
    params = [float(v) for v in params]
    if len(params) > 3:
        raise ValueError("at most 3 activation parameters")
    a = _abi.MoeActivation()
    a.kind = _abi.ACTIVATIONS[kind]
    a.n_params = len(params)
    for i, v in enumerate(params):
        a.params[i] = v
    return a


# ------------------------------------------------------------------ grouped matmul
def gmm_forward(x: torch.Tensor, w: torch.Tensor, group_list: torch.Tensor, *, epilogue: int = 0,
                clip: float = 0.0, y: Optional[torch.Tensor] = None, h_save: Optional[torch.Tensor] = None,
                activation=None, w_transposed: bool = False, ws: Optional[Workspace] = None,
                stream=None) -> torch.Tensor:
    """y = grouped x @ w (epilogue 1: SwiGLU over the [gate | up] halves; or,
    with `activation` = (kind, params), that gated activation).  With
    w_transposed, w is [E, N, K] (each expert's weight transposed)."""
    _dtype(x, BF16, "x")
    _dtype(w, BF16, "w")
    _dtype(group_list, torch.int64, "group_list")
    M, K = x.shape
    E, K2, N = w.shape
    if w_transposed:
        K2, N = N, K2
    if K2 != K:
        raise ValueError("x and w disagree on K")
    out_cols = N // 2 if (epilogue == _abi.MOE_EPILOGUE_SWIGLU or activation is not None) else N
    if y is None:
        y = torch.empty(M, out_cols, dtype=BF16, device=x.device)
    wsp = _ws(ws, gmm_workspace_size(M, K, N, E), x.device)
    if activation is not None or w_transposed:
        if activation is None and epilogue == _abi.MOE_EPILOGUE_SWIGLU:
            activation = ("swiglu", [clip])
        a = C.byref(_act(activation)) if activation is not None else None
        _check(_lib().gmm_forward_act(_ptr(x), _ptr(w), _ptr(group_list), M, K, N, E, a, int(bool(w_transposed)),
                                      _ptr(y), _ptr(h_save), wsp.ptr, wsp.nbytes, _stream(stream)), "gmm_forward_act")
        return y
    _check(_lib().gmm_forward(_ptr(x), _ptr(w), _ptr(group_list), M, K, N, E, int(epilogue), float(clip),
                              _ptr(y), _ptr(h_save), wsp.ptr, wsp.nbytes, _stream(stream)), "gmm_forward")
    return y


def gmm_forward_gather_act(x: torch.Tensor, sorted_flat: torch.Tensor, k: int, w: torch.Tensor,
                           group_list: torch.Tensor, activation=("swiglu", ()), *, M: Optional[int] = None,
                           y: Optional[torch.Tensor] = None, w_transposed: bool = False,
                           ws: Optional[Workspace] = None, stream=None) -> torch.Tensor:
    """The gate_up GMM with its activation over rows gathered from x: row r of
    the grouped operand is token sorted_flat[r] // k (M rows, default
    len(sorted_flat)); returns y [M, N/2]."""
    _dtype(x, BF16, "x")
    _dtype(sorted_flat, torch.int32, "sorted_flat")
    _dtype(w, BF16, "w")
    _dtype(group_list, torch.int64, "group_list")
    T, K = x.shape
    M = sorted_flat.shape[0] if M is None else M
    E, K2, N = w.shape
    if w_transposed:
        K2, N = N, K2
    if K2 != K:
        raise ValueError("x and w disagree on K")
    if y is None:
        y = torch.empty(M, N // 2, dtype=BF16, device=x.device)
    wsp = _ws(ws, gmm_workspace_size(M, K, N, E), x.device)
    _check(_lib().gmm_forward_gather_act(_ptr(x), _ptr(sorted_flat), T, k, _ptr(w), _ptr(group_list), M, K, N, E,
                                         C.byref(_act(activation)), int(bool(w_transposed)), _ptr(y), wsp.ptr,
                                         wsp.nbytes, _stream(stream)), "gmm_forward_gather_act")
    return y


def moe_expert_mlp_workspace_size(T, k, E) -> int:
    return int(_lib().moe_expert_mlp_workspace_size(T, k, E))


def moe_expert_mlp_forward(x: torch.Tensor, sorted_flat: torch.Tensor, group_list: torch.Tensor, w1: torch.Tensor,
                           w2: torch.Tensor, k: int, activation=("swiglu", ()), *, a=None, y2=None,
                           ws: Optional[Workspace] = None, stream=None):
    """Both expert matmuls in one launch, the gate_up rows gathered from x:
    returns (a [T*k, I], y2 [T*k, H])."""
    for t, n in ((x, "x"), (w1, "w1"), (w2, "w2")):
        _dtype(t, BF16, n)
    _dtype(sorted_flat, torch.int32, "sorted_flat")
    _dtype(group_list, torch.int64, "group_list")
    T, H = x.shape
    E, I = w2.shape[0], w2.shape[1]
    if a is None:
        a = torch.empty(T * k, I, dtype=BF16, device=x.device)
    if y2 is None:
        y2 = torch.empty(T * k, H, dtype=BF16, device=x.device)
    wsp = _ws(ws, moe_expert_mlp_workspace_size(T, k, E), x.device)
    _check(_lib().moe_expert_mlp_forward(_ptr(x), _ptr(sorted_flat), _ptr(group_list), _ptr(w1), _ptr(w2), T, H, I, E,
                                         k, C.byref(_act(activation)), _ptr(a), _ptr(y2), wsp.ptr, wsp.nbytes,
                                         _stream(stream)), "moe_expert_mlp_forward")
    return a, y2


def gmm_forward_combine_workspace_size(T, k, M, N) -> int:
    return int(_lib().gmm_forward_combine_workspace_size(T, k, M, N))


def gmm_forward_combine(a: torch.Tensor, w: torch.Tensor, group_list: torch.Tensor, row_id_map: torch.Tensor,
                        sorted_flat: torch.Tensor, topk_w: torch.Tensor, *, y: Optional[torch.Tensor] = None,
                        w_transposed: bool = False, ws: Optional[Workspace] = None, stream=None) -> torch.Tensor:
    """The down GMM fused with the weighted top-k combine: y [T, N] =
    moe_unpermute(gmm_forward(a, w), row_id_map, topk_w), bit for bit."""
    _dtype(a, BF16, "a")
    _dtype(w, BF16, "w")
    _dtype(group_list, torch.int64, "group_list")
    _dtype(row_id_map, torch.int32, "row_id_map")
    _dtype(sorted_flat, torch.int32, "sorted_flat")
    _dtype(topk_w, torch.float32, "topk_w")
    M, K = a.shape
    T, k = topk_w.shape
    E = w.shape[0]
    N = w.shape[1] if w_transposed else w.shape[2]
    if y is None:
        y = torch.empty(T, N, dtype=BF16, device=a.device)
    wsp = _ws(ws, gmm_forward_combine_workspace_size(T, k, M, N), a.device)
    _check(_lib().gmm_forward_combine(_ptr(a), _ptr(w), _ptr(group_list), _ptr(row_id_map), _ptr(sorted_flat),
                                      _ptr(topk_w), T, k, M, K, N, E, int(bool(w_transposed)), _ptr(y), wsp.ptr,
                                      wsp.nbytes, _stream(stream)), "gmm_forward_combine")
    return y


def gmm_backward(x: torch.Tensor, w: torch.Tensor, group_list: torch.Tensor, dy: torch.Tensor, *,
                 need_dx: bool = True, need_dw: bool = True, dx=None, dw=None, w_transposed: bool = False,
                 ws: Optional[Workspace] = None, stream=None):
    """Returns (dx [M, K] or None, dw [E, K, N] or None); with w_transposed, w
    is [E, N, K] and so is dw."""
    _dtype(x, BF16, "x")
    _dtype(w, BF16, "w")
    _dtype(dy, BF16, "dy")
    M, K = x.shape
    E, N = w.shape[0], dy.shape[1]
    if need_dx and dx is None:
        dx = torch.empty(M, K, dtype=BF16, device=x.device)
    if need_dw and dw is None:
        dw = torch.empty(E, *((N, K) if w_transposed else (K, N)), dtype=BF16, device=x.device)
    wsp = _ws(ws, gmm_workspace_size(M, K, N, E), x.device)
    _check(_lib().gmm_backward_ex(_ptr(x), _ptr(w), _ptr(group_list), _ptr(dy), M, K, N, E, int(bool(w_transposed)),
                                  _ptr(dx if need_dx else None), _ptr(dw if need_dw else None),
                                  wsp.ptr, wsp.nbytes, _stream(stream)), "gmm_backward_ex")
    return (dx if need_dx else None), (dw if need_dw else None)


def gmm_backward_dx_swiglu(dy: torch.Tensor, w: torch.Tensor, group_list: torch.Tensor, h: torch.Tensor,
                           clip: float = 0.0, *, dh=None, activation=None, w_transposed: bool = False,
                           ws: Optional[Workspace] = None, stream=None) -> torch.Tensor:
    """dh = SwiGLU (or `activation`) gradient of h given dA = grouped dy @ w^T,
    in one pass (dA is not stored)."""
    for t, n in ((dy, "dy"), (w, "w"), (h, "h")):
        _dtype(t, BF16, n)
    M, N = dy.shape
    E = w.shape[0]
    K = w.shape[2] if w_transposed else w.shape[1]
    if dh is None:
        dh = torch.empty(M, 2 * K, dtype=BF16, device=dy.device)
    wsp = _ws(ws, gmm_workspace_size(M, K, N, E), dy.device)
    if activation is not None or w_transposed:
        activation = activation if activation is not None else ("swiglu", [clip])
        _check(_lib().gmm_backward_dx_act(_ptr(dy), _ptr(w), _ptr(group_list), _ptr(h), M, K, N, E,
                                          C.byref(_act(activation)), int(bool(w_transposed)), _ptr(dh), wsp.ptr,
                                          wsp.nbytes, _stream(stream)), "gmm_backward_dx_act")
        return dh
    _check(_lib().gmm_backward_dx_swiglu(_ptr(dy), _ptr(w), _ptr(group_list), _ptr(h), M, K, N, E, float(clip),
                                         _ptr(dh), wsp.ptr, wsp.nbytes, _stream(stream)), "gmm_backward_dx_swiglu")
    return dh


# ------------------------------------------------------------------ combine side
def moe_unpermute(y_perm, row_id_map, topk_w, T: int, k: int, *, y=None, ws=None, stream=None):
    H = y_perm.shape[1]
    _dtype(y_perm, BF16, "y_perm")
    _dtype(topk_w, torch.float32, "topk_w")
    if y is None:
        y = torch.empty(T, H, dtype=BF16, device=y_perm.device)
    wsp = _ws(ws, moe_unpermute_workspace_size(), y_perm.device)
    _check(_lib().moe_unpermute(_ptr(y_perm), _ptr(row_id_map), _ptr(topk_w), T, H, k, _ptr(y),
                                wsp.ptr, wsp.nbytes, _stream(stream)), "moe_unpermute")
    return y


def moe_unpermute_backward(dy, y_perm, row_id_map, topk_w, k: int, *, dy_perm=None, dprobs=None,
                           need_dprobs: bool = True, ws=None, stream=None):
    T, H = dy.shape
    _dtype(dy, BF16, "dy")
    _dtype(y_perm, BF16, "y_perm")
    if dy_perm is None:
        dy_perm = torch.empty(T * k, H, dtype=BF16, device=dy.device)
    if need_dprobs and dprobs is None:
        dprobs = torch.empty(T, k, dtype=torch.float32, device=dy.device)
    wsp = _ws(ws, moe_unpermute_workspace_size(), dy.device)
    _check(_lib().moe_unpermute_backward(_ptr(dy), _ptr(y_perm), _ptr(row_id_map), _ptr(topk_w), T, H, k,
                                         _ptr(dy_perm), _ptr(dprobs if need_dprobs else None),
                                         wsp.ptr, wsp.nbytes, _stream(stream)), "moe_unpermute_backward")
    return dy_perm, (dprobs if need_dprobs else None)


def moe_permute_backward(dx_perm, row_id_map, T: int, k: int, *, dx=None, ws=None, stream=None):
    H = dx_perm.shape[1]
    _dtype(dx_perm, BF16, "dx_perm")
    if dx is None:
        dx = torch.empty(T, H, dtype=BF16, device=dx_perm.device)
    wsp = _ws(ws, moe_unpermute_workspace_size(), dx_perm.device)
    _check(_lib().moe_permute_backward(_ptr(dx_perm), _ptr(row_id_map), T, H, k, _ptr(dx),
                                       wsp.ptr, wsp.nbytes, _stream(stream)), "moe_permute_backward")
    return dx


def moe_swiglu_backward(h, da, clip: float = 0.0, *, dh=None, activation=None, ws=None, stream=None):
    rows, I2 = h.shape
    _dtype(h, BF16, "h")
    _dtype(da, BF16, "da")
    if dh is None:
        dh = torch.empty_like(h)
    wsp = _ws(ws, moe_unpermute_workspace_size(), h.device)
    if activation is not None:
        _check(_lib().moe_activation_backward(_ptr(h), _ptr(da), rows, I2 // 2, C.byref(_act(activation)), _ptr(dh),
                                              wsp.ptr, wsp.nbytes, _stream(stream)), "moe_activation_backward")
        return dh
    _check(_lib().moe_swiglu_backward(_ptr(h), _ptr(da), rows, I2 // 2, float(clip), _ptr(dh),
                                      wsp.ptr, wsp.nbytes, _stream(stream)), "moe_swiglu_backward")
    return dh


# ------------------------------------------------------------------ whole layer
class LayerSaved:
    """Device buffers the layer forward fills for the backward."""

    def __init__(self, T, H, I, E, k, device="cuda"):
        R = T * k
        self.x_perm = torch.empty(R, H, dtype=BF16, device=device)
        self.h = torch.empty(R, 2 * I, dtype=BF16, device=device)
        self.a = torch.empty(R, I, dtype=BF16, device=device)
        self.y2 = torch.empty(R, H, dtype=BF16, device=device)
        self.row_id_map = torch.empty(R, dtype=torch.int32, device=device)
        self.sorted_flat = torch.empty(R, dtype=torch.int32, device=device)
        self.group_list = torch.empty(E, dtype=torch.int64, device=device)

    def struct(self) -> _abi.MoeLayerSaved:
        return _abi.MoeLayerSaved(*(t.data_ptr() for t in (self.x_perm, self.h, self.a, self.y2, self.row_id_map,
                                                             self.sorted_flat, self.group_list)))


def moe_layer_forward(x, topk_ids, topk_w, w1, w2, clip: float = 0.0, *, saved: Optional[LayerSaved] = None,
                      y=None, activation=None, w_flags: int = 0, ws: Optional[Workspace] = None, stream=None):
    """w_flags: bit 0 = w1 stored [E, 2I, H], bit 1 = w2 stored [E, H, I]."""
    T, H = x.shape
    E = w1.shape[0]
    I2 = w1.shape[1] if w_flags & 1 else w1.shape[2]
    I = I2 // 2
    k = topk_ids.shape[1]
    for t, n in ((x, "x"), (w1, "w1"), (w2, "w2")):
        _dtype(t, BF16, n)
    _dtype(topk_ids, torch.int32, "topk_ids")
    _dtype(topk_w, torch.float32, "topk_w")
    if y is None:
        y = torch.empty(T, H, dtype=BF16, device=x.device)
    wsp = _ws(ws, moe_layer_workspace_size(T, H, I, E, k), x.device)
    sv = C.byref(saved.struct()) if saved is not None else None
    if activation is not None or w_flags:
        activation = activation if activation is not None else ("swiglu", [clip])
        _check(_lib().moe_layer_forward_act(_ptr(x), _ptr(topk_ids), _ptr(topk_w), _ptr(w1), _ptr(w2), T, H, I, E,
                                            k, C.byref(_act(activation)), int(w_flags), _ptr(y), sv, wsp.ptr,
                                            wsp.nbytes, _stream(stream)), "moe_layer_forward_act")
        return y
    _check(_lib().moe_layer_forward(_ptr(x), _ptr(topk_ids), _ptr(topk_w), _ptr(w1), _ptr(w2), T, H, I, E, k,
                                    float(clip), _ptr(y), sv, wsp.ptr, wsp.nbytes, _stream(stream)),
           "moe_layer_forward")
    return y


def moe_layer_backward(dy, topk_w, w1, w2, saved: LayerSaved, clip: float = 0.0, *, dx=None, dw1=None, dw2=None,
                       dprobs=None, activation=None, w_flags: int = 0, ws: Optional[Workspace] = None, stream=None):
    """dw1 and dw2 come in the weights' layouts (w_flags as for moe_layer_forward)."""
    T, H = dy.shape
    E = w1.shape[0]
    I2 = w1.shape[1] if w_flags & 1 else w1.shape[2]
    I = I2 // 2
    k = topk_w.shape[1]
    dev = dy.device
    dx = torch.empty(T, H, dtype=BF16, device=dev) if dx is None else dx
    dw1 = torch.empty_like(w1) if dw1 is None else dw1
    dw2 = torch.empty_like(w2) if dw2 is None else dw2
    dprobs = torch.empty(T, k, dtype=torch.float32, device=dev) if dprobs is None else dprobs
    wsp = _ws(ws, moe_layer_workspace_size(T, H, I, E, k), dev)
    if activation is not None or w_flags:
        activation = activation if activation is not None else ("swiglu", [clip])
        _check(_lib().moe_layer_backward_act(_ptr(dy), _ptr(topk_w), _ptr(w1), _ptr(w2), C.byref(saved.struct()),
                                             T, H, I, E, k, C.byref(_act(activation)), int(w_flags), _ptr(dx),
                                             _ptr(dw1), _ptr(dw2), _ptr(dprobs), wsp.ptr, wsp.nbytes,
                                             _stream(stream)), "moe_layer_backward_act")
        return dx, dw1, dw2, dprobs
    _check(_lib().moe_layer_backward(_ptr(dy), _ptr(topk_w), _ptr(w1), _ptr(w2), C.byref(saved.struct()),
                                     T, H, I, E, k, float(clip), _ptr(dx), _ptr(dw1), _ptr(dw2), _ptr(dprobs),
                                     wsp.ptr, wsp.nbytes, _stream(stream)), "moe_layer_backward")
    return dx, dw1, dw2, dprobs


# ------------------------------------------------------------------ MXFP8 forward (include/moe_mx.h)
U8 = torch.uint8


def _fmt(name):
    if name not in _abi.FP8_FORMATS:
        raise ValueError("unknown MX element format %r (e4m3, e5m2 or e2m1)" % (name,))
    return _abi.FP8_FORMATS[name]


def _code_cols(K: int, fmt: str) -> int:
    """Bytes per row of K codes: E2M1 packs two per byte."""
    return K // 2 if fmt == "e2m1" else K


def activation_format(x_fmt: str) -> str:
    """The element type gmm_forward_mx quantises the activation to: the tokens'
    fp8 type, or E4M3 after E2M1 tokens ("MegaMoE", A4W4-FP 量化场景)."""
    return "e4m3" if x_fmt == "e2m1" else x_fmt


def moe_mx_quantize(x, fmt: str = "e4m3", *, q=None, scales=None, ws: Optional[Workspace] = None, stream=None):
    """Q_MX of each row of x [rows, K] bf16: (q [rows, K] uint8 codes, or
    [rows, K/2] packed E2M1, scales [rows, K/32] uint8 E8M0 codes)."""
    _dtype(x, BF16, "x")
    rows, K = x.shape
    q = torch.empty(rows, _code_cols(K, fmt), dtype=U8, device=x.device) if q is None else q
    scales = torch.empty(rows, K // 32, dtype=U8, device=x.device) if scales is None else scales
    _dtype(q, U8, "q")
    _dtype(scales, U8, "scales")
    w = _ws(ws, int(_lib().moe_mx_quantize_workspace_size()), x.device)
    _check(_lib().moe_mx_quantize(_ptr(x), rows, K, _fmt(fmt), _ptr(q), _ptr(scales), w.ptr, w.nbytes,
                                  _stream(stream)), "moe_mx_quantize")
    return q, scales


def moe_permute_mx(x, topk_ids, E: int, fmt: str = "e4m3", *, out=None, ws: Optional[Workspace] = None, stream=None):
    """moe_permute whose gathered rows leave quantised: returns (x_q [T*k, H] uint8
    ([T*k, H/2] packed E2M1), x_scales [T*k, H/32] uint8, group_list, row_id_map,
    sorted_flat)."""
    _dtype(x, BF16, "x")
    _dtype(topk_ids, torch.int32, "topk_ids")
    T, k = topk_ids.shape
    H = x.shape[1]
    dev = topk_ids.device
    if out is None:
        out = (torch.empty(T * k, _code_cols(H, fmt), dtype=U8, device=dev),
               torch.empty(T * k, H // 32, dtype=U8, device=dev),
               torch.empty(E, dtype=torch.int64, device=dev), torch.empty(T * k, dtype=torch.int32, device=dev),
               torch.empty(T * k, dtype=torch.int32, device=dev))
    x_q, x_s, group_list, row_id_map, sorted_flat = out
    w = _ws(ws, moe_permute_workspace_size(T, k, E), dev)
    _check(_lib().moe_permute_mx(_ptr(x), _ptr(topk_ids), T, H, k, E, _fmt(fmt), _ptr(x_q), _ptr(x_s),
                                 _ptr(group_list), _ptr(row_id_map), _ptr(sorted_flat), w.ptr, w.nbytes,
                                 _stream(stream)), "moe_permute_mx")
    return x_q, x_s, group_list, row_id_map, sorted_flat


def gmm_forward_mx(x_q, x_scales, w_q, w_scales, group_list, *, x_fmt: str = "e4m3", w_fmt: str = "e4m3",
                   activation=None, y=None, a_q=None, a_scales=None, h_save=None, ws: Optional[Workspace] = None,
                   stream=None):
    """Block-scaled grouped matmul: x_q [M, K] / x_scales [M, K/32], w_q [E, N, K] /
    w_scales [E, N, K/32] (uint8 codes; E2M1 operands packed, K/2 bytes a row).
    Without an activation returns y [M, N] bf16; with one returns
    (a_q [M, N/2], a_scales [M, N/64]) in activation_format(x_fmt)."""
    M = x_q.shape[0]
    K = x_scales.shape[1] * 32
    E, N, _ = w_q.shape
    for t, n in ((x_q, "x_q"), (x_scales, "x_scales"), (w_q, "w_q"), (w_scales, "w_scales")):
        _dtype(t, U8, n)
    _dtype(group_list, torch.int64, "group_list")
    dev = x_q.device
    act = C.byref(_act(activation)) if activation is not None else None
    if activation is None:
        y = torch.empty(M, N, dtype=BF16, device=dev) if y is None else y
    else:
        a_q = torch.empty(M, N // 2, dtype=U8, device=dev) if a_q is None else a_q
        a_scales = torch.empty(M, N // 64, dtype=U8, device=dev) if a_scales is None else a_scales
    w = _ws(ws, int(_lib().gmm_mx_workspace_size(M, K, N, E)), dev)
    _check(_lib().gmm_forward_mx(_ptr(x_q), _ptr(x_scales), _ptr(w_q), _ptr(w_scales), _ptr(group_list), M, K, N,
                                 E, _fmt(x_fmt), _fmt(w_fmt), act, _ptr(y), _ptr(a_q), _ptr(a_scales),
                                 _ptr(h_save), w.ptr, w.nbytes, _stream(stream)), "gmm_forward_mx")
    return y if activation is None else (a_q, a_scales)


def moe_layer_mx_workspace_size(T, H, I, E, k) -> int:
    return int(_lib().moe_layer_mx_workspace_size(T, H, I, E, k))


def moe_layer_forward_mx(x, topk_ids, topk_w, w1_q, w1_scales, w2_q, w2_scales, *, x_fmt: str = "e4m3",
                         w_fmt: str = "e4m3", activation="swiglu", y=None, ws: Optional[Workspace] = None,
                         stream=None):
    """MX layer forward (A8W8-FP, A8W4-FP with w_fmt "e2m1", A4W4-FP with x_fmt and
    w_fmt "e2m1"): w1_q [E, 2I, H], w2_q [E, H, I] codes (E2M1 packed, half the
    last dimension) with their [.., K/32] E8M0 scales; returns y [T, H] bf16."""
    T, H = x.shape
    E, I2, _ = w1_q.shape
    I = I2 // 2
    k = topk_ids.shape[1]
    _dtype(x, BF16, "x")
    _dtype(topk_ids, torch.int32, "topk_ids")
    _dtype(topk_w, torch.float32, "topk_w")
    for t, n in ((w1_q, "w1_q"), (w1_scales, "w1_scales"), (w2_q, "w2_q"), (w2_scales, "w2_scales")):
        _dtype(t, U8, n)
    y = torch.empty(T, H, dtype=BF16, device=x.device) if y is None else y
    wsp = _ws(ws, moe_layer_mx_workspace_size(T, H, I, E, k), x.device)
    _check(_lib().moe_layer_forward_mx(_ptr(x), _ptr(topk_ids), _ptr(topk_w), _ptr(w1_q), _ptr(w1_scales),
                                       _ptr(w2_q), _ptr(w2_scales), T, H, I, E, k, _fmt(x_fmt), _fmt(w_fmt),
                                       C.byref(_act(activation)), _ptr(y), wsp.ptr, wsp.nbytes, _stream(stream)),
           "moe_layer_forward_mx")
    return y
