"""CPU oracle for the routed-expert MoE hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU baseline
and its ``--impl reference`` arm) may import or run this module.  The product
path (``moe_routed_expert_gb300``) never imports it and shares no code with it.

What it is: a plain, slow, obviously-correct restatement of what the method
computes, in float64, using numpy's matmul as the only library step.  It
rounds to bfloat16 (round to nearest even) exactly where the method stores a
bf16 tensor; pass ``store=None`` to any function to get the exact real-number
result instead (the pins in ``tests/test_oracle_pins.py`` use that for finite
differences and adjoint identities).

Sources (page title, then section):

* [GMM] "NPU Training Operators - GMM":
  - section "算子语义" (operator semantics): the eager per-group loop, the
    worked example (pairs -> group_list [1,2,0,2]), the row-to-weight table
    with the empty bucket 3:3, and the backward formulas
    grad_input_e = grad_output_e @ W_e^T, grad_weight_e = X_e^T @ grad_output_e;
  - section "Qwen3.5 MoE 路径": the routed-expert pipeline
    permute -> histc -> GMM(gate_up) -> SwiGLU -> GMM(down) -> unpermute(probs),
    and the two GMM shapes;
  - section "验证项": bf16 tolerance rtol=1e-2, atol=1e-2.
* [MegaMoE] "MegaMoE" (ops-transformer operator doc):
  - "计算公式 / 激活函数公式": sigma, SiLU, the clip value c (unset or 0 means
    +inf), G_c = min(G, c), U_c = clip(U, -c, c), swiglu = SiLU(G_c) * U_c,
    swiglustep = min(SiLU(G), c) * U_c, swigluoai = G_c * sigma(alpha G_c) *
    (U_c + beta), situglu = beta tanh(G / beta) * sigma(G) * L(U) with
    L(U) = U, or linear_beta tanh(U / linear_beta) when linear_beta is given;
  - "参数说明" (activation, activation_params): the parameter lists and their
    defaults (clamp: no clip; alpha 1.702; swigluoai beta 1.0; situglu beta
    1.0 and no linear_beta);
  - "A16W16 非量化场景": EP Dispatch (row(i,k), rows of X_e stacked in any fixed
    order), Expert Compute (H_e = X_e W1[e], split into gate G and up U,
    Y_e = A_e W2[e]), Token Combine (y_i = sum_k w_k Y_{e_ik}[row(i,k)],
    outputs stacked in input order);
  - "A8W8-FP 量化场景": gate is the first N/2 columns of W1, up the last N/2.
* [MegaBlocks-03] "03 · grouped GEMM path", section 4.3: activation backward
  from the saved GMM output (activation recomputed in backward).
* [PermuteGrad] "CANN ops-transformer 算子详解 MoeTokenPermuteWithRoutingMapGrad":
  section 2.3 (token gradient: zeros, then index-add of the permuted rows,
  accumulate semantics), section 2.2 (probs gradient), section 6.2 (per output
  token walk its topK slots, skip -1, accumulate).
* [Qwen3.5-MoE inference] "Qwen3.5-MoE 在 NPU 上的推理性能优化实践", section 3.3
  (gate_proj and up_proj merged into one weight; GMM -> swiglu -> GMM ->
  finalize_routing).

Readings taken where the pages leave a step open (each is also listed in the
design notes of the repository):

1. group_list holds per-expert counts (int64); boundaries are its cumsum.
2. "any fixed order" of rows inside an expert: ascending flat slot index
   f = t*k + j (a stable counting sort).  This reproduces the worked example.
3. gate = first I columns of H, up = last I columns.
4. The clip gradient passes at the kink: d/dG is taken as 1 where G <= c and
   d/dU as 1 where -c <= U <= c.
5. Combine, token gradient and probs gradient accumulate in higher precision
   and round once.
6. The probs gradient has the shape of topk_w, [T, k].
7. A topk id of -1 marks an unused slot: it is not counted, adds nothing to
   y and gets a zero probs gradient.
8. Expert weights are [E, K, N] row-major.
9. The pre-activation H is rounded to bf16 before SwiGLU (the unfused
   pipeline stores the gate_up GMM output, then applies swiglu).
10. Rounding is round-to-nearest-even everywhere.
11. dW is stored in bf16, like W; an empty group's dW is zero.
12. The activation variants' gradients (the pages give none: MegaMoE is an
    inference operator) are the derivatives of their formulas, taking every
    min / clip kink as passing the gradient (as in reading 4): swiglustep's
    min(SiLU(G), c) passes d/dG where SiLU(G) <= c.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "round_to_bf16", "bf16_bits_to_f64", "f64_to_bf16_bits",
    "histogram", "exclusive_scan", "stable_counting_sort", "moe_permute",
    "expert_matmul", "gmm_forward", "gmm_backward",
    "sigmoid", "silu", "clip_bound", "swiglu", "swiglu_backward",
    "ACTIVATIONS", "activation", "gated_activation", "gated_activation_backward",
    "moe_unpermute", "moe_unpermute_backward", "moe_permute_backward",
    "moe_layer_forward", "moe_layer_backward",
]


# --------------------------------------------------------------------------
# bfloat16 storage
# --------------------------------------------------------------------------
def round_to_bf16(v):
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 has float32's 8-bit exponent and 8 significant bits.  A value
    v = m * 2**e (0.5 <= |m| < 1) lies on a grid of spacing 2**(e-8); below the
    normal range (2**-126) the grid spacing stays 2**-133 (subnormals).
    Results of magnitude 2**128 or more overflow to +-inf; inf and nan pass
    through unchanged.  Works through the array in chunks of 2**20 values.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.empty_like(v)
    src, dst = v.reshape(-1), out.reshape(-1)
    step = 1 << 20
    with np.errstate(invalid="ignore", over="ignore"):
        for s in range(0, src.size, step):
            c = src[s:s + step]
            _, e = np.frexp(c)
            q = np.maximum(e - 8, -133)
            r = np.ldexp(np.round(np.ldexp(c, -q)), q)  # np.round: half to even
            dst[s:s + step] = np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, c), r)
    return out if v.ndim else out[()]


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Raw bfloat16 bits (uint16) -> float64 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, np.float64)
    src, dst = b.reshape(-1), out.reshape(-1)
    step = 1 << 22
    for s in range(0, src.size, step):
        dst[s:s + step] = (src[s:s + step].astype(np.uint32) << 16).view(np.float32)
    return out


def f64_to_bf16_bits(v) -> np.ndarray:
    """float64 -> raw bfloat16 bits, rounding to nearest even first."""
    r = round_to_bf16(v).astype(np.float32)  # exact: every bf16 value is a float32 value
    return (r.view(np.uint32) >> 16).astype(np.uint16)


def _store(store, v):
    return v if store is None else store(v)


# --------------------------------------------------------------------------
# S1-S4: permute (dispatch) -- [GMM] "算子语义" worked example and
# "Qwen3.5 MoE 路径" (permute, tokens_per_expert = histc); [MegaMoE] EP Dispatch
# --------------------------------------------------------------------------
def _check_ids(topk_ids, E):
    ids = np.asarray(topk_ids)
    if ids.ndim != 2:
        raise ValueError("topk_ids must be [T, k]")
    if ids.size and (ids.min() < -1 or ids.max() >= E):
        raise ValueError("topk ids must lie in [-1, E)")
    return ids


def histogram(topk_ids, E: int) -> np.ndarray:
    """counts[e] = number of slots (t, j) with topk_ids[t, j] == e; -1 slots are skipped."""
    ids = _check_ids(topk_ids, E).ravel()
    counts = np.zeros(E, dtype=np.int64)
    for e in ids.tolist():
        if e >= 0:
            counts[e] += 1
    return counts


def exclusive_scan(counts) -> np.ndarray:
    """offsets[e] = sum of counts[e'] for e' < e; offsets[E] = total rows.

    Expert e owns rows [offsets[e], offsets[e+1]); an empty expert owns an
    empty range and leaves every later offset unchanged."""
    counts = np.asarray(counts, dtype=np.int64)
    off = np.zeros(len(counts) + 1, dtype=np.int64)
    run = 0
    for e, n in enumerate(counts.tolist()):
        if n < 0:
            raise ValueError("negative group count")
        off[e] = run
        run += n
    off[len(counts)] = run
    return off


def stable_counting_sort(topk_ids, E: int):
    """Dispatch row map.  Walk the flat slots f = t*k + j in ascending order;
    slot f with expert e gets row offsets[e] + (number of earlier slots with the
    same expert).

    Returns (row_id_map[T*k] int32 with -1 for unused slots,
             sorted_flat[R] int32 = inverse map row -> flat slot,
             counts[E] int64, offsets[E+1] int64)."""
    ids = _check_ids(topk_ids, E)
    counts = histogram(ids, E)
    off = exclusive_scan(counts)
    nxt = off[:-1].copy()
    flat = ids.ravel().tolist()
    row_id_map = np.full(len(flat), -1, dtype=np.int32)
    sorted_flat = np.zeros(int(off[-1]), dtype=np.int32)
    for f, e in enumerate(flat):
        if e < 0:
            continue
        r = nxt[e]
        nxt[e] += 1
        row_id_map[f] = r
        sorted_flat[r] = f
    return row_id_map, sorted_flat, counts, off


def moe_permute(x, topk_ids, E: int):
    """x_perm[row] = x[token of the slot that owns row].

    Returns (x_perm[R, H], group_list[E] counts, row_id_map[T*k], sorted_flat[R])."""
    ids = _check_ids(topk_ids, E)
    k = ids.shape[1]
    row_id_map, sorted_flat, counts, _ = stable_counting_sort(ids, E)
    x = np.asarray(x)
    x_perm = x[sorted_flat.astype(np.int64) // k]
    return x_perm, counts, row_id_map, sorted_flat


# --------------------------------------------------------------------------
# Grouped matmul -- [GMM] "算子语义" (eager loop, backward formulas)
# --------------------------------------------------------------------------
def expert_matmul(x_rows, w_e, store=round_to_bf16):
    """One group's product x_rows @ w_e, exact in float64, then stored."""
    return _store(store, np.asarray(x_rows, np.float64) @ np.asarray(w_e, np.float64))


def _group_bounds(group_list, M):
    counts = np.asarray(group_list, dtype=np.int64)
    off = exclusive_scan(counts)
    if off[-1] != M:
        raise ValueError("sum(group_list) must equal the number of rows")
    return off


def gmm_forward(x, w, group_list, store=round_to_bf16):
    """y[s:e] = x[s:e] @ w[g] for each group g with rows [s, e) (eager loop)."""
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    off = _group_bounds(group_list, x.shape[0])
    y = np.zeros((x.shape[0], w.shape[2]))
    for g in range(w.shape[0]):
        s, e = off[g], off[g + 1]
        if e > s:
            y[s:e] = _store(store, x[s:e] @ w[g])
    return y


def gmm_backward(x, w, group_list, dy, store=round_to_bf16):
    """grad_input_g = dy_g @ w[g]^T and grad_weight_g = x_g^T @ dy_g per group;
    an empty group's grad_weight is zero."""
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    dy = np.asarray(dy, np.float64)
    off = _group_bounds(group_list, x.shape[0])
    dx = np.zeros_like(x)
    dw = np.zeros_like(w)
    for g in range(w.shape[0]):
        s, e = off[g], off[g + 1]
        if e > s:
            dx[s:e] = _store(store, dy[s:e] @ w[g].T)
            dw[g] = _store(store, x[s:e].T @ dy[s:e])
    return dx, dw


# --------------------------------------------------------------------------
# SwiGLU with clip -- [MegaMoE] "激活函数公式" (swiglu) and Expert Compute step 2
# --------------------------------------------------------------------------
def sigmoid(z):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-np.asarray(z, np.float64)))


def silu(z):
    z = np.asarray(z, np.float64)
    return z * sigmoid(z)


def clip_bound(clip) -> float:
    """The clip value c: unset (None) or 0 means +inf; negative is invalid."""
    if clip is None or clip == 0:
        return np.inf
    if clip < 0:
        raise ValueError("clip must be >= 0")
    return float(clip)


def swiglu(h, clip=None, store=round_to_bf16):
    """h = [G | U] (gate = first half of the columns, up = second half);
    A = SiLU(min(G, c)) * clip(U, -c, c)."""
    h = np.asarray(h, np.float64)
    I = h.shape[1] // 2
    c = clip_bound(clip)
    g, u = h[:, :I], h[:, I:]
    gc = np.minimum(g, c)
    uc = np.clip(u, -c, c)
    return _store(store, silu(gc) * uc)


def swiglu_backward(h, da, clip=None, store=round_to_bf16):
    """Gradient of swiglu w.r.t. h = [G | U]:
    dG = dA * U_c * SiLU'(G_c) * [G <= c],  dU = dA * SiLU(G_c) * [-c <= U <= c],
    SiLU'(z) = sigma(z) * (1 + z * (1 - sigma(z)))."""
    h = np.asarray(h, np.float64)
    da = np.asarray(da, np.float64)
    I = h.shape[1] // 2
    c = clip_bound(clip)
    g, u = h[:, :I], h[:, I:]
    gc = np.minimum(g, c)
    uc = np.clip(u, -c, c)
    s = sigmoid(gc)
    dsilu = s * (1.0 + gc * (1.0 - s))
    dg = da * uc * dsilu * (g <= c)
    du = da * silu(gc) * ((u >= -c) & (u <= c))
    return _store(store, np.concatenate([dg, du], axis=1))


# --------------------------------------------------------------------------
# Combine (unpermute) and its gradients -- [MegaMoE] Token Combine;
# [PermuteGrad] sections 2.2, 2.3, 6.2
# --------------------------------------------------------------------------
# Gated activation variants ([MegaMoE] 激活函数公式, 参数说明)
# --------------------------------------------------------------------------
ACTIVATIONS = ("swiglu", "swiglustep", "swigluoai", "situglu")


def activation(kind="swiglu", params=()):
    """The activation and its parameters from the pages' (activation,
    activation_params) pair, with the defaults of an empty list:
    swiglu / swiglustep take [] or [clamp]; swigluoai [] or [clamp, alpha,
    beta] (alpha 1.702, beta 1.0); situglu [], [beta] or [beta, linear_beta]
    (beta 1.0, no linear_beta).  clamp 0 or absent means no clip."""
    if kind not in ACTIVATIONS:
        raise ValueError("unknown activation %r" % (kind,))
    params = [float(v) for v in params]
    a = dict(kind=kind, c=np.inf, alpha=1.702, beta=1.0, linear_beta=None)
    if kind in ("swiglu", "swiglustep", "swigluoai"):
        if len(params) not in ((0, 1) if kind != "swigluoai" else (0, 3)):
            raise ValueError("bad activation_params for %s" % kind)
        if params:
            a["c"] = clip_bound(params[0])
        if kind == "swigluoai" and params:
            a["alpha"], a["beta"] = params[1], params[2]
    else:
        if len(params) > 2:
            raise ValueError("bad activation_params for situglu")
        if params:
            a["beta"] = params[0]
        if len(params) == 2:
            a["linear_beta"] = params[1]
        if not (a["beta"] > 0 and np.isfinite(a["beta"])):
            raise ValueError("situglu beta must be finite and > 0")
        if a["linear_beta"] is not None and not (a["linear_beta"] > 0 and np.isfinite(a["linear_beta"])):
            raise ValueError("situglu linear_beta must be finite and > 0")
    return a


def gated_activation(h, act, store=round_to_bf16):
    """A from h = [G | U] for one of the four activations (formulas above)."""
    h = np.asarray(h, np.float64)
    I = h.shape[1] // 2
    g, u = h[:, :I], h[:, I:]
    c, kind = act["c"], act["kind"]
    if kind == "swiglu":
        v = silu(np.minimum(g, c)) * np.clip(u, -c, c)
    elif kind == "swiglustep":
        v = np.minimum(silu(g), c) * np.clip(u, -c, c)
    elif kind == "swigluoai":
        gc = np.minimum(g, c)
        v = gc * sigmoid(act["alpha"] * gc) * (np.clip(u, -c, c) + act["beta"])
    else:
        b, lb = act["beta"], act["linear_beta"]
        lu = u if lb is None else lb * np.tanh(u / lb)
        v = b * np.tanh(g / b) * sigmoid(g) * lu
    return _store(store, v)


def gated_activation_backward(h, da, act, store=round_to_bf16):
    """dH = [dG | dU] for gated_activation, the derivative of each formula
    (reading 12 for the kinks)."""
    h = np.asarray(h, np.float64)
    da = np.asarray(da, np.float64)
    I = h.shape[1] // 2
    g, u = h[:, :I], h[:, I:]
    c, kind = act["c"], act["kind"]
    in_u = (u >= -c) & (u <= c)
    uc = np.clip(u, -c, c)
    if kind == "swiglu":
        gc = np.minimum(g, c)
        s = sigmoid(gc)
        dg = da * uc * s * (1.0 + gc * (1.0 - s)) * (g <= c)
        du = da * silu(gc) * in_u
    elif kind == "swiglustep":
        s = sigmoid(g)
        sg = silu(g)
        dg = da * uc * s * (1.0 + g * (1.0 - s)) * (sg <= c)
        du = da * np.minimum(sg, c) * in_u
    elif kind == "swigluoai":
        al, be = act["alpha"], act["beta"]
        gc = np.minimum(g, c)
        s = sigmoid(al * gc)
        dg = da * (uc + be) * (s + al * gc * s * (1.0 - s)) * (g <= c)
        du = da * gc * s * in_u
    else:
        b, lb = act["beta"], act["linear_beta"]
        t = np.tanh(g / b)
        s = sigmoid(g)
        if lb is None:
            lu, dlu = u, np.ones_like(u)
        else:
            tl = np.tanh(u / lb)
            lu, dlu = lb * tl, 1.0 - tl * tl
        dg = da * lu * ((1.0 - t * t) * s + b * t * s * (1.0 - s))
        du = da * b * t * s * dlu
    return _store(store, np.concatenate([dg, du], axis=1))


# --------------------------------------------------------------------------
def _slots(row_id_map, T, k):
    r = np.asarray(row_id_map, dtype=np.int64).reshape(T, k)
    return r


def moe_unpermute(y_perm, row_id_map, topk_w, T: int, k: int, store=round_to_bf16):
    """y[t] = sum over j of topk_w[t, j] * y_perm[row(t, j)], skipping unused slots."""
    y_perm = np.asarray(y_perm, np.float64)
    w = np.asarray(topk_w, np.float64).reshape(T, k)
    rows = _slots(row_id_map, T, k)
    y = np.zeros((T, y_perm.shape[1]))
    for j in range(k):
        ok = rows[:, j] >= 0
        y[ok] += w[ok, j, None] * y_perm[rows[ok, j]]
    return _store(store, y)


def moe_unpermute_backward(dy, y_perm, row_id_map, topk_w, T: int, k: int, store=round_to_bf16):
    """Gradients of the combine:
    dy_perm[row(t, j)] = topk_w[t, j] * dy[t],
    dprobs[t, j] = <dy[t], y_perm[row(t, j)]> (0 for an unused slot).
    Rows of dy_perm owned by no slot stay zero.  dprobs is returned unrounded
    (it is a float32 output)."""
    dy = np.asarray(dy, np.float64)
    y_perm = np.asarray(y_perm, np.float64)
    w = np.asarray(topk_w, np.float64).reshape(T, k)
    rows = _slots(row_id_map, T, k)
    dy_perm = np.zeros_like(y_perm)
    dprobs = np.zeros((T, k))
    for j in range(k):
        ok = rows[:, j] >= 0
        dy_perm[rows[ok, j]] = w[ok, j, None] * dy[ok]
        dprobs[ok, j] = np.sum(dy[ok] * y_perm[rows[ok, j]], axis=1)
    return _store(store, dy_perm), dprobs


def moe_permute_backward(dx_perm, row_id_map, T: int, k: int, store=round_to_bf16):
    """Token gradient: start from zeros and add each slot's permuted row back to
    its token (index-add), dx[t] = sum over j of dx_perm[row(t, j)]."""
    dx_perm = np.asarray(dx_perm, np.float64)
    rows = _slots(row_id_map, T, k)
    dx = np.zeros((T, dx_perm.shape[1]))
    for j in range(k):
        ok = rows[:, j] >= 0
        dx[ok] += dx_perm[rows[ok, j]]
    return _store(store, dx)


# --------------------------------------------------------------------------
# The routed-expert layer -- [GMM] "Qwen3.5 MoE 路径"; [MegaMoE] A16W16
# --------------------------------------------------------------------------
def moe_layer_forward(x, topk_ids, topk_w, w1, w2, clip=None, store=round_to_bf16, act=None):
    """permute -> GMM(gate_up) -> SwiGLU -> GMM(down) -> weighted combine.

    `act` (from activation()) selects another gated activation; by default
    SwiGLU with the clip `clip`.
    Returns (y[T, H], saved) where saved holds the tensors the backward needs:
    x_perm, group_list, row_id_map, sorted_flat, h (pre-activation), a, y2."""
    ids = np.asarray(topk_ids)
    T, k = ids.shape
    E = np.asarray(w1).shape[0]
    x_perm, counts, row_id_map, sorted_flat = moe_permute(np.asarray(x, np.float64), ids, E)
    h = gmm_forward(x_perm, w1, counts, store)
    a = swiglu(h, clip, store) if act is None else gated_activation(h, act, store)
    y2 = gmm_forward(a, w2, counts, store)
    y = moe_unpermute(y2, row_id_map, topk_w, T, k, store)
    saved = dict(x_perm=x_perm, group_list=counts, row_id_map=row_id_map, sorted_flat=sorted_flat,
                 h=h, a=a, y2=y2)
    return y, saved


def moe_layer_backward(dy, saved, topk_w, w1, w2, clip=None, store=round_to_bf16, act=None):
    """Backward of moe_layer_forward.  Returns (dx[T, H], dw1, dw2, dprobs[T, k])."""
    dy = np.asarray(dy, np.float64)
    T = dy.shape[0]
    rows = np.asarray(saved["row_id_map"])
    k = rows.size // T
    counts = saved["group_list"]
    dy2, dprobs = moe_unpermute_backward(dy, saved["y2"], rows, topk_w, T, k, store)
    da, dw2 = gmm_backward(saved["a"], w2, counts, dy2, store)
    dh = swiglu_backward(saved["h"], da, clip, store) if act is None else \
        gated_activation_backward(saved["h"], da, act, store)
    dx_perm, dw1 = gmm_backward(saved["x_perm"], w1, counts, dh, store)
    dx = moe_permute_backward(dx_perm, rows, T, k, store)
    return dx, dw1, dw2, dprobs
