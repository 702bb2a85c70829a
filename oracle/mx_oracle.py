"""CPU oracle for the MXFP8 routed-expert forward (A8W8-FP) -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU baseline
and its ``--impl reference`` arm) may import or run this module.  The product
path never imports it and shares no code with it.

What it is: the MX quantised forward written out in float64, element formats
decoded from their bit fields and rounding done by explicit nearest-value
search, so that a reader can check each step by eye.

Sources (page title, then section):

* [MegaMoE] "MegaMoE" (ops-transformer operator doc), "A8W8-FP 量化场景":
  - stage 1: the rows gathered per expert are quantised with Q_MX, group size
    32 along the row, a shared exponent per group, elements in FLOAT8_E5M2 or
    FLOAT8_E4M3FN, scales in FLOAT8_E8M0;
  - stage 2: G_e = DQ(X_e) DQ(W1_e^G), U_e = DQ(X_e) DQ(W1_e^U) (gate = the
    first N/2 output columns of weight1, up = the last N/2),
    A_e = Activation(G_e, U_e), then Q_MX(A_e) in the same element type as
    stage 1;
  - stage 3: O_e = DQ(A_e) DQ(W2_e);
  - stage 4: Y[i] = sum_k W[i, k] O[pi(i, k)] (the A16W16 combine).
* [MegaMoE] "约束说明", MXFP constraints: weight1 is (E, 2I, H), weight2 is
  (E, H, I) (each output channel a row of K contiguous elements);
  weightScales1 is (E, 2I, ceil(H/64), 2) and weightScales2 is
  (E, H, ceil(I/64), 2), both E8M0, i.e. one scale per 32 elements of K; the
  scales of a pre-quantised x are (BS, ceil(H/32)).
* [MegaMoE] "A8W4-FP 量化场景": the same four stages with MXFP4 (FLOAT4_E2M1)
  weights for both matmuls and E4M3 tokens / activations (the data flow BF16 ->
  MXFP8 E4M3 -> A8W4 GMM1 -> MXFP8 E4M3 -> A8W4 GMM2 -> BF16).
* [MegaMoE] "A4W4-FP 量化场景": the tokens are quantised to MXFP4 (E2M1
  elements, E8M0 scales, groups of 32), GMM1 multiplies MXFP4 tokens by MXFP4
  weights, the activation is quantised to MXFP8 E4M3 (not E2M1, to keep the
  second matmul's precision), so GMM2 is A8W4 (the data flow BF16 -> MXFP4
  E2M1 -> A4W4 GMM1 -> MXFP8 E4M3 -> A8W4 GMM2 -> BF16).
* The element and scale formats are the ones the pages name by type:
  FLOAT8_E4M3FN (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
  infinities, S.1111.111 is NaN, largest finite 448), FLOAT8_E5M2 (bias 15,
  2 mantissa bits, IEEE-style infinities and NaNs, largest finite 57344),
  FLOAT4_E2M1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit, no
  infinities or NaNs: 0, 0.5, 1, 1.5, 2, 3, 4, 6) and FLOAT8_E8M0 (an
  unsigned biased exponent: 2^(code - 127), 0xFF is NaN).

Readings taken where the pages leave a step open (also listed in the design
notes of the repository):

M1. "Extract a shared exponent" is read as the usual MX rule: for a group of
    32 values with largest magnitude amax, the scale is
    X = 2^(floor(log2 amax) - emax), emax = 8 for E4M3 and 15 for E5M2 (the
    exponent of the element type's largest power of two), clamped to
    [2^-127, 2^127].  amax = 0 gives 2^-127 (code 0); a group holding an
    infinity or a NaN gets the NaN scale (code 0xFF) and NaN elements.
M2. Each element is x / X rounded to the nearest value of the element type,
    ties to the even code, saturating to the largest finite magnitude
    (x / X may reach 2^(emax+1), above 448 and 57344).
M3. The gate / up pre-activations are rounded to bf16 before the activation
    (as in the A16W16 path); the activation's fp output is quantised directly.
M4. O_e is stored in bf16 and combined like the A16W16 path's expert outputs.
M5. K of both matmuls (H and I) is a multiple of 128.
M6. E2M1 has no NaN: a NaN value encodes as the largest magnitude (code 7,
    or 15 with its sign); emax = 2 (the largest power of two, 4).  Codes are
    held one per array element here; the CUDA path takes them packed two per
    byte (a layout, see workloads.pack_fp4).
M7. The activation is quantised in the tokens' element type when that is an
    fp8 type, and in E4M3 when the tokens are E2M1 (the A4W4-FP rule above).
    Other pairings of token and weight types than the pages' four scenarios
    follow the same stages (the matmul takes any pair).
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import (activation, gated_activation, gmm_forward, moe_permute, moe_unpermute, round_to_bf16)

__all__ = [
    "FP8_FORMATS", "fp8_decode", "fp8_encode", "fp8_finite_values", "e8m0_decode",
    "mx_quantize", "mx_dequantize", "mx_gmm", "mx_layer_forward", "activation_format", "MX_BLOCK",
]

MX_BLOCK = 32

# ebits, mbits, bias; emax = exponent of the largest finite power of two.
FP8_FORMATS = {
    "e4m3": dict(bits=8, ebits=4, mbits=3, bias=7, emax=8, max=448.0, nan_code=0x7F),
    "e5m2": dict(bits=8, ebits=5, mbits=2, bias=15, emax=15, max=57344.0, nan_code=0x7F),
    "e2m1": dict(bits=4, ebits=2, mbits=1, bias=1, emax=2, max=6.0, nan_code=0x7),
}


def _fmt(fmt):
    if fmt not in FP8_FORMATS:
        raise ValueError("unknown fp8 format %r" % (fmt,))
    return FP8_FORMATS[fmt]


def fp8_decode(codes, fmt) -> np.ndarray:
    """Value of each code (8 bits, or the low 4 bits for e2m1), from its sign /
    exponent / mantissa fields."""
    f = _fmt(fmt)
    c = np.asarray(codes, dtype=np.int64)
    eb, mb, bias = f["ebits"], f["mbits"], f["bias"]
    sign = np.where((c >> (f["bits"] - 1)) & 1, -1.0, 1.0)
    e = (c >> mb) & ((1 << eb) - 1)
    m = c & ((1 << mb) - 1)
    frac = m / float(1 << mb)
    val = np.where(e == 0, frac * 2.0 ** (1 - bias), (1.0 + frac) * np.exp2(e.astype(np.float64) - bias))
    top = (1 << eb) - 1
    if fmt == "e2m1":
        pass                                             # every code is finite
    elif fmt == "e4m3":
        val = np.where((e == top) & (m == (1 << mb) - 1), np.nan, val)
    else:
        val = np.where((e == top) & (m == 0), np.inf, val)
        val = np.where((e == top) & (m != 0), np.nan, val)
    return sign * val


def fp8_finite_values(fmt):
    """(codes, values) of the non-negative finite codes, ascending."""
    codes = np.arange(1 << (_fmt(fmt)["bits"] - 1))
    vals = fp8_decode(codes, fmt)
    keep = np.isfinite(vals)
    return codes[keep], vals[keep]


def fp8_encode(v, fmt) -> np.ndarray:
    """Nearest code to each value (ties to the even code), saturating to the
    largest finite magnitude; NaN gives the format's NaN code.  The sign is
    carried over, so -0.0 and negative values that round to zero give 0x80."""
    f = _fmt(fmt)
    v = np.asarray(v, dtype=np.float64)
    codes, vals = fp8_finite_values(fmt)
    mag = np.minimum(np.abs(v), f["max"])
    hi = np.searchsorted(vals, mag, side="left")          # first value >= mag
    hi = np.minimum(hi, len(vals) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - vals[lo]
    d_hi = vals[hi] - mag
    exact = vals[hi] == mag
    pick_hi = exact | (d_hi < d_lo) | ((d_hi == d_lo) & (codes[hi] % 2 == 0))
    out = np.where(pick_hi, codes[hi], codes[lo])
    out = out | np.where(np.signbit(v), 1 << (f["bits"] - 1), 0)
    out = np.where(np.isnan(v), f["nan_code"], out)
    return out.astype(np.uint8)


def e8m0_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.int64)
    return np.where(c == 255, np.nan, np.exp2(c.astype(np.float64) - 127))


def mx_quantize(x, fmt):
    """Q_MX over the last axis (a multiple of 32): (codes uint8 [..., K],
    scale codes uint8 [..., K/32])."""
    f = _fmt(fmt)
    x = np.asarray(x, dtype=np.float64)
    K = x.shape[-1]
    if K % MX_BLOCK:
        raise ValueError("the quantised axis must be a multiple of %d" % MX_BLOCK)
    xb = x.reshape(x.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    amax = np.max(np.abs(xb), axis=-1)                   # NaN if the group holds one
    finite = np.isfinite(amax)
    safe = np.where(finite & (amax > 0), amax, 1.0)
    _, ex = np.frexp(safe)                               # safe = m 2^ex, m in [0.5, 1)
    e = (ex - 1) - f["emax"]                             # floor(log2 amax) - emax
    e = np.where(amax > 0, e, -127)
    e = np.clip(e, -127, 127)
    scale_codes = np.where(finite, e + 127, 255).astype(np.uint8)
    scaled = xb / np.exp2(np.where(finite, e, 0))[..., None]
    q = fp8_encode(scaled, fmt)
    q = np.where(finite[..., None], q, np.uint8(f["nan_code"]))
    return q.reshape(x.shape).astype(np.uint8), scale_codes


def mx_dequantize(codes, scale_codes, fmt) -> np.ndarray:
    """DQ_MX: element value times its group's scale (the element values looked
    up in the table of all 256 decoded codes)."""
    v = fp8_decode(np.arange(256), fmt)[np.asarray(codes, dtype=np.int64)]
    K = v.shape[-1]
    vb = v.reshape(v.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    s = e8m0_decode(scale_codes)[..., None]
    return (vb * s).reshape(v.shape)


def mx_gmm(xq, xs, wq, ws, group_list, x_fmt, w_fmt, store=round_to_bf16):
    """DQ(X_e) DQ(W_e)^T per group: xq [M, K], xs [M, K/32], wq [E, N, K],
    ws [E, N, K/32] (one output channel per row of W_e)."""
    x = mx_dequantize(xq, xs, x_fmt)
    w = mx_dequantize(wq, ws, w_fmt)
    return gmm_forward(x, np.ascontiguousarray(np.transpose(w, (0, 2, 1))), group_list, store)


def activation_format(x_fmt):
    """The element type of the quantised activation (reading M7)."""
    return "e4m3" if x_fmt == "e2m1" else x_fmt


def mx_layer_forward(x, topk_ids, topk_w, w1q, w1s, w2q, w2s, x_fmt="e4m3", w_fmt="e4m3", act=None,
                     store=round_to_bf16):
    """The four stages of the A8W8-FP / A8W4-FP / A4W4-FP forward on one device.

    x: bf16-valued [T, H]; w1q [E, 2I, H] / w1s [E, 2I, H/32]; w2q [E, H, I] /
    w2s [E, H, I/32].  Returns (y [T, H], saved) with the intermediates."""
    x = np.asarray(x, dtype=np.float64)
    T, H = x.shape
    E = w1q.shape[0]
    k = np.asarray(topk_ids).shape[1]
    act = activation("swiglu") if act is None else act
    x_perm, group_list, row_id_map, _ = moe_permute(x, topk_ids, E)
    xq, xs = mx_quantize(x_perm, x_fmt)                                   # stage 1
    h = mx_gmm(xq, xs, w1q, w1s, group_list, x_fmt, w_fmt, store=round_to_bf16)  # G | U, bf16 (M3)
    a = gated_activation(h, act, store=None)                              # stage 2
    a_fmt = activation_format(x_fmt)
    aq, as_ = mx_quantize(a, a_fmt)
    o = mx_gmm(aq, as_, w2q, w2s, group_list, a_fmt, w_fmt, store=store)  # stage 3 (M4)
    y = moe_unpermute(o, row_id_map, topk_w, T, k, store=store)           # stage 4
    saved = dict(x_perm=x_perm, group_list=group_list, row_id_map=row_id_map, xq=xq, xs=xs,
                 h=h, a=a, aq=aq, as_=as_, o=o)
    return y, saved
