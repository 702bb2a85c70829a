"""Parity of the MX forward (include/moe_mx.h: A8W8-FP, A8W4-FP, A4W4-FP) with
the oracle.

- Q_MX of bf16 rows is exact arithmetic (an exponent read off amax, a scaling
  by a power of two, one rounding), so codes and scales must match the oracle
  bit for bit, special groups included (zeros, signed zeros, saturation,
  infinities and NaNs, the clamped smallest scale).
- The block-scaled grouped matmul: the same dequantised operands on both
  sides, fp32 accumulation against float64, bf16 output: within the pages'
  rtol = atol = 1e-2.
- The activation + Q_MX epilogue: H (saved in bf16) against the oracle within
  tolerance; the codes and scales against the oracle's activation and Q_MX of
  the GPU's own H.  Those are decisions taken from an activation the GPU
  evaluates in fp32 and the oracle in float64, so a code may differ where the
  exact value lies within a relative 1e-5 of a rounding midpoint (and a scale
  where amax lies that close to a power of two); every other code must match.
- The layer: equal, bit for bit, to the chain of the single calls; its y
  against the oracle's four stages within tolerance; at full prefill size on
  a sample of tokens.
"""
import numpy as np
import pytest

import oracle as O
from oracle import mx_oracle as X
from tests._util import assert_close, dev, dev_bf16, f64, host_f64
from workloads import (WORKLOADS, fp8_codes, e8m0_codes, layer_inputs, mx_layer_weights, mx_weight, normal_bf16,
                       pack_fp4, unpack_fp4)

pytestmark = pytest.mark.gpu

FMTS = ["e4m3", "e5m2", "e2m1"]


def np_u8(t):
    return t.detach().cpu().numpy().astype(np.uint8)


def w_dev(codes, fmt):
    """Codes as the CUDA path takes them: E2M1 packed two per byte."""
    return dev(pack_fp4(codes) if fmt == "e2m1" else codes)


def codes_of(t, fmt):
    """A device tensor of codes as one code per byte."""
    return unpack_fp4(np_u8(t)) if fmt == "e2m1" else np_u8(t)


def special_rows(fmt, K=256):
    """bf16-valued rows that hit every branch of Q_MX."""
    f = X.FP8_FORMATS[fmt]
    rows = np.zeros((8, K))
    rows[1, :32] = -0.0
    rows[1, 32:64] = 2.0 ** -130                       # subnormal amax: clamped scale
    rows[2, :32] = np.linspace(-1, 1, 32) * 1.9        # saturates at the top
    rows[2, 32] = np.inf
    rows[3, 64] = np.nan
    rows[3, 65] = 1.0
    rows[4, :] = 2.0 ** 120 * np.sign(np.sin(np.arange(K)))
    rows[5, :] = 2.0 ** -120 * np.cos(np.arange(K))
    rows[6, :32] = f["max"] * 2.0 ** -f["emax"] * np.array([(-1) ** i for i in range(32)])  # exactly max
    rows[7, :] = np.arange(K) - K / 2
    return O.round_to_bf16(rows)


def compare_quant(q_gpu, s_gpu, x, fmt):
    q, s = X.mx_quantize(x, fmt)
    assert np.array_equal(s_gpu, s)
    if fmt == "e2m1":        # no NaN code: every code of a NaN-scaled group is 7 on both sides
        assert np.array_equal(q_gpu, q)
        return
    nan_group = np.repeat(s == 255, 32, axis=-1)
    assert np.array_equal(q_gpu[~nan_group], q[~nan_group])
    assert np.all(np.isnan(X.fp8_decode(q_gpu[nan_group], fmt)))


@pytest.mark.parametrize("fmt", FMTS)
def test_mx_quantize_bit_exact(fmt):
    import moe_routed_expert_gb300 as M
    rng = np.random.default_rng(21)
    x = f64(normal_bf16(rng, (300, 1056))) * np.exp2(rng.integers(-40, 40, (300, 1)))
    x = O.round_to_bf16(x)
    xs = np.concatenate([x[:, :256], special_rows(fmt)], axis=0)
    for arr in (x, xs):
        bits = O.f64_to_bf16_bits(arr)
        q, s = M.moe_mx_quantize(dev_bf16(bits), fmt)
        compare_quant(codes_of(q, fmt), np_u8(s), arr, fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_permute_mx(fmt):
    import moe_routed_expert_gb300 as M
    wl = WORKLOADS["layer_prefill_t4096"].with_tokens(300)
    inp = layer_inputs(wl, tokens=300, with_weights=False)
    ids = inp["topk_ids"].copy()
    ids[5, 3] = -1                                            # an unused slot
    x = inp["x"]
    xq, xs, gl, rmap, sflat = M.moe_permute_mx(dev_bf16(x), dev(ids), wl.E, fmt)
    x_perm, counts, rmap_o, sflat_o = O.moe_permute(f64(x), ids, wl.E)
    R = int(counts.sum())
    assert np.array_equal(host_f64(gl), counts)
    assert np.array_equal(host_f64(rmap), rmap_o)
    assert np.array_equal(host_f64(sflat)[:R], sflat_o)
    compare_quant(codes_of(xq, fmt)[:R], np_u8(xs)[:R], x_perm, fmt)


def mx_gmm_case(rng, E, K, N, counts, x_fmt, w_fmt):
    M_ = int(np.sum(counts))
    centre = 127 - 4 - int(round(0.5 * np.log2(K)))
    xq = fp8_codes(rng, (M_, K), x_fmt)
    xs = e8m0_codes(rng, (M_, K // 32), 123)
    wq, ws = mx_weight(rng, E, N, K, w_fmt)
    return xq, xs, wq, ws, np.asarray(counts, np.int64), centre


GMM_CASES = [
    # E, K, N, counts, x_fmt, w_fmt
    (4, 256, 384, [37, 0, 200, 91], "e4m3", "e4m3"),      # empty group, ragged rows, ragged column tile
    (4, 256, 256, [1, 130, 0, 255], "e5m2", "e5m2"),
    (3, 640, 512, [129, 64, 0], "e4m3", "e5m2"),          # mixed element types, 5 K blocks over a 4-stage ring
    (8, 1024, 768, [300, 0, 17, 512, 1, 0, 90, 256], "e4m3", "e4m3"),
    # MXFP4 (E2M1) weights, "A8W4-FP 量化场景"
    (4, 256, 384, [37, 0, 200, 91], "e4m3", "e2m1"),
    (3, 640, 512, [129, 64, 0], "e5m2", "e2m1"),
    (8, 1024, 768, [300, 0, 17, 512, 1, 0, 90, 256], "e4m3", "e2m1"),
    # MXFP4 tokens, "A4W4-FP 量化场景" (and E2M1 tokens with fp8 weights)
    (4, 256, 384, [37, 0, 200, 91], "e2m1", "e2m1"),
    (3, 640, 512, [129, 64, 0], "e2m1", "e4m3"),
    (8, 1024, 768, [300, 0, 17, 512, 1, 0, 90, 256], "e2m1", "e2m1"),
]


@pytest.mark.parametrize("case", GMM_CASES, ids=lambda c: "E%d_K%d_N%d_%s_%s" % (c[0], c[1], c[2], c[4], c[5]))
def test_gmm_forward_mx_plain(case):
    import moe_routed_expert_gb300 as M
    E, K, N, counts, xf, wf = case
    rng = np.random.default_rng(31)
    xq, xs, wq, ws, gl, _ = mx_gmm_case(rng, E, K, N, counts, xf, wf)
    wsp = M.Workspace(256)
    y = M.gmm_forward_mx(w_dev(xq, xf), dev(xs), w_dev(wq, wf), dev(ws), dev(gl), x_fmt=xf, w_fmt=wf, ws=wsp)
    assert M.read_status(wsp) == 0
    want = X.mx_gmm(xq, xs, wq, ws, gl, xf, wf)
    assert_close("y", y, want)


# Groups of a few rows, as in decode: many 128-row tiles that hold 0-12 rows,
# one group over 32 rows, empty groups; N = 384 leaves a ragged 256-column tile.
SMALL_COUNTS = [3, 0, 1, 40, 2, 0, 7, 1, 0, 5, 2, 2, 0, 9, 1, 1, 0, 3, 4, 0, 1, 1, 6, 0, 2, 3, 0, 1, 2, 0, 0, 12]
# A sparse batch (about 6 rows per expert) with one group of 300 rows among 63
# small ones: three 128-row tiles for the big group, the last ragged.
SPARSE_BIG_GROUP = [300] + [2, 0, 1, 3] * 15 + [0, 5, 1]
SWAP_CASES = [("e4m3", "e4m3", 384), ("e5m2", "e5m2", 256), ("e4m3", "e2m1", 384), ("e2m1", "e2m1", 384)]


@pytest.mark.parametrize("xf,wf,N", SWAP_CASES)
def test_gmm_forward_mx_small_groups_plain(xf, wf, N):
    import moe_routed_expert_gb300 as M
    rng = np.random.default_rng(51)
    E, K = len(SMALL_COUNTS), 512
    xq, xs, wq, ws, gl, _ = mx_gmm_case(rng, E, K, N, SMALL_COUNTS, xf, wf)
    wsp = M.Workspace(256)
    y = M.gmm_forward_mx(w_dev(xq, xf), dev(xs), w_dev(wq, wf), dev(ws), dev(gl), x_fmt=xf, w_fmt=wf, ws=wsp)
    assert M.read_status(wsp) == 0
    assert_close("y", y, X.mx_gmm(xq, xs, wq, ws, gl, xf, wf))


@pytest.mark.parametrize("xf,wf", [("e4m3", "e4m3"), ("e5m2", "e5m2"), ("e4m3", "e2m1"), ("e2m1", "e2m1")])
@pytest.mark.parametrize("act", [("swiglu", (7.0,)), ("situglu", (1.0, 2.0))], ids=lambda a: a[0])
def test_gmm_forward_mx_small_groups_activation(act, xf, wf):
    import torch
    import moe_routed_expert_gb300 as M
    rng = np.random.default_rng(52)
    E, K, I = len(SMALL_COUNTS), 256, 256
    xq, xs, wq, ws, gl, _ = mx_gmm_case(rng, E, K, 2 * I, SMALL_COUNTS, xf, wf)
    Mr = int(sum(SMALL_COUNTS))
    h = torch.empty(Mr, 2 * I, dtype=torch.bfloat16, device="cuda")
    wsp = M.Workspace(256)
    aq, as_ = M.gmm_forward_mx(w_dev(xq, xf), dev(xs), w_dev(wq, wf), dev(ws), dev(gl), x_fmt=xf, w_fmt=wf,
                               activation=(act[0], list(act[1])), h_save=h, ws=wsp)
    assert M.read_status(wsp) == 0
    assert_close("h", h, X.mx_gmm(xq, xs, wq, ws, gl, xf, wf))
    check_act_codes(np_u8(aq), np_u8(as_), host_f64(h), O.activation(act[0], act[1]), X.activation_format(xf))


def check_act_codes(aq, as_, h_gpu, act, fmt, rel=1e-5, abs_a=2e-6):
    """Codes and scales against Q_MX(activation(H)) of the GPU's own H: a
    decision may differ only where the exact value sits within the fp32
    evaluation's error of its boundary: rel |a| + abs_a in activation units.
    The absolute term covers situglu, whose tanh, computed as
    1 - 2 / (1 + e^{2z}), has an absolute rather than relative error (4.8e-7
    against float64 in a float32 emulation over 2e5 draws; up to 1e-4
    relative for |a| > 1e-3)."""
    a = O.gated_activation(h_gpu, act, store=None)
    q_ref, s_ref = X.mx_quantize(a, fmt)
    f = X.FP8_FORMATS[fmt]
    rows, I = a.shape
    ab = a.reshape(rows, I // 32, 32)
    amax = np.max(np.abs(ab), axis=2)
    # scales: equal, or amax within rel of a power of two
    near_pow2 = np.abs(amax / np.exp2(np.round(np.log2(np.maximum(amax, 1e-300)))) - 1.0) < rel
    bad_s = (as_ != s_ref) & ~near_pow2
    assert not np.any(bad_s), "scale mismatch away from a power of two at %s" % (np.argwhere(bad_s)[:5],)
    # codes, checked against the GPU's own scale: the GPU's value must be the
    # nearest one, or tie with it within rel
    X_gpu = np.repeat(X.e8m0_decode(as_), 32, axis=1)
    r = np.clip(a / X_gpu, -f["max"], f["max"])
    best = X.fp8_decode(X.fp8_encode(r, fmt), fmt)
    got = X.fp8_decode(aq, fmt)
    d_best, d_got = np.abs(best - r), np.abs(got - r)
    ok = (aq == X.fp8_encode(r, fmt)) | (d_got - d_best <= rel * np.abs(r) + abs_a / X_gpu)
    assert np.all(ok), "code mismatch away from a midpoint at %s" % (np.argwhere(~ok)[:5],)
    frac = np.mean(aq != q_ref)
    assert frac < 1e-3, frac


ACT_CASES = [
    ("swiglu", ()), ("swiglu", (7.0,)), ("swiglustep", (1.5,)), ("swigluoai", (7.0, 1.702, 1.0)),
    ("situglu", (1.0, 2.0)),
]


@pytest.mark.parametrize("fmt,wfmt", [("e4m3", "e4m3"), ("e5m2", "e5m2"), ("e4m3", "e2m1"), ("e2m1", "e2m1")])
@pytest.mark.parametrize("act", ACT_CASES, ids=lambda a: a[0] + "".join("_%g" % v for v in a[1]))
def test_gmm_forward_mx_activation(act, fmt, wfmt):
    import torch
    import moe_routed_expert_gb300 as M
    rng = np.random.default_rng(41)
    E, K, I = 4, 384, 256
    counts = [70, 0, 257, 33]
    xq, xs, wq, ws, gl, _ = mx_gmm_case(rng, E, K, 2 * I, counts, fmt, wfmt)
    Mr = int(sum(counts))
    h = torch.empty(Mr, 2 * I, dtype=torch.bfloat16, device="cuda")
    wsp = M.Workspace(256)
    aq, as_ = M.gmm_forward_mx(w_dev(xq, fmt), dev(xs), w_dev(wq, wfmt), dev(ws), dev(gl), x_fmt=fmt, w_fmt=wfmt,
                               activation=(act[0], list(act[1])), h_save=h, ws=wsp)
    assert M.read_status(wsp) == 0
    want_h = X.mx_gmm(xq, xs, wq, ws, gl, fmt, wfmt)
    assert_close("h", h, want_h)
    check_act_codes(np_u8(aq), np_u8(as_), host_f64(h), O.activation(act[0], act[1]), X.activation_format(fmt))


def gpu_mx_chain(inp, wts, wl, fmt, act, wfmt=None):
    """The layer as the chain of single calls."""
    import moe_routed_expert_gb300 as M
    wfmt = wfmt or fmt
    x, ids, tw = dev_bf16(inp["x"]), dev(inp["topk_ids"]), dev(inp["topk_w"])
    wsc = M.Workspace(M.moe_permute_workspace_size(wl.T, wl.k, wl.E))
    xq, xs, gl, rmap, _ = M.moe_permute_mx(x, ids, wl.E, fmt, ws=wsc)
    import torch
    h = torch.empty(xq.shape[0], 2 * wl.I, dtype=torch.bfloat16, device="cuda")
    aq, as_ = M.gmm_forward_mx(xq, xs, w_dev(wts["w1_q"], wfmt), dev(wts["w1_s"]), gl, x_fmt=fmt, w_fmt=wfmt,
                               activation=act, h_save=h, ws=wsc)
    o = M.gmm_forward_mx(aq, as_, w_dev(wts["w2_q"], wfmt), dev(wts["w2_s"]), gl, x_fmt=X.activation_format(fmt),
                         w_fmt=wfmt, ws=wsc)
    y = M.moe_unpermute(o, rmap, tw, wl.T, wl.k, ws=wsc)
    assert M.read_status(wsc) == 0
    return dict(xq=xq, xs=xs, gl=gl, rmap=rmap, h=h, aq=aq, as_=as_, o=o, y=y)


@pytest.mark.parametrize("fmt,wfmt", [("e4m3", "e4m3"), ("e5m2", "e5m2"), ("e4m3", "e2m1"), ("e2m1", "e2m1")])
def test_layer_mx_small(fmt, wfmt):
    check_layer_mx(fmt, wfmt, T=96, H=256, E=8, k=4, I=128)


@pytest.mark.parametrize("fmt,wfmt", [("e4m3", "e4m3"), ("e4m3", "e2m1")])
def test_layer_mx_max_experts(fmt, wfmt):
    """1024 experts (the library's limit): 1280 routed slots take the
    multi-block index pass and leave about 29% of the experts empty."""
    check_layer_mx(fmt, wfmt, T=160, H=256, E=1024, k=8, I=128)


@pytest.mark.parametrize("fmt,wfmt", [("e4m3", "e4m3"), ("e4m3", "e2m1"), ("e2m1", "e2m1")])
def test_layer_mx_one_token(fmt, wfmt):
    """A single token routed to 8 of 8 experts: one row per expert, every tile
    of both block-scaled matmuls holding one valid row."""
    check_layer_mx(fmt, wfmt, T=1, H=256, E=8, k=8, I=128)


def check_layer_mx(fmt, wfmt, **shape):
    """moe_layer_forward_mx against the chain of single calls (bit-identical),
    each step of the chain on its own input, and y end to end."""
    import moe_routed_expert_gb300 as M
    wl = WORKLOADS["layer_prefill_mx_t4096"]
    wl = type(wl)(**{**wl.__dict__, **shape, "mx": fmt, "w_mx": wfmt})
    inp = layer_inputs(wl, with_weights=False)
    wts = mx_layer_weights(wl)
    act = ("swiglu", [7.0])
    wsp = M.Workspace(M.moe_layer_mx_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.k))
    y = M.moe_layer_forward_mx(dev_bf16(inp["x"]), dev(inp["topk_ids"]), dev(inp["topk_w"]),
                               w_dev(wts["w1_q"], wfmt), dev(wts["w1_s"]), w_dev(wts["w2_q"], wfmt),
                               dev(wts["w2_s"]), x_fmt=fmt, w_fmt=wfmt, activation=act, ws=wsp)
    assert M.read_status(wsp) == 0
    ch = gpu_mx_chain(inp, wts, wl, fmt, act, wfmt)
    assert np.array_equal(host_f64(y), host_f64(ch["y"]))
    # each step on the GPU's own input to it
    oa = O.activation(*act)
    x_perm, counts, rmap_o, _ = O.moe_permute(f64(inp["x"]), inp["topk_ids"], wl.E)
    R = int(counts.sum())
    xq = codes_of(ch["xq"], fmt)
    compare_quant(xq[:R], np_u8(ch["xs"])[:R], x_perm, fmt)
    assert_close("h", ch["h"], X.mx_gmm(xq, np_u8(ch["xs"]), wts["w1_q"], wts["w1_s"], counts, fmt, wfmt))
    afmt = X.activation_format(fmt)
    check_act_codes(np_u8(ch["aq"]), np_u8(ch["as_"]), host_f64(ch["h"]), oa, afmt)
    o_want = X.mx_gmm(np_u8(ch["aq"]), np_u8(ch["as_"]), wts["w2_q"], wts["w2_s"], counts, afmt, wfmt)
    assert_close("o", ch["o"], o_want)
    # end to end
    y_want, _ = X.mx_layer_forward(f64(inp["x"]), inp["topk_ids"], inp["topk_w"], wts["w1_q"], wts["w1_s"],
                                   wts["w2_q"], wts["w2_s"], fmt, wfmt, oa)
    assert_close("y", y, y_want)


@pytest.mark.parametrize("name", ["layer_prefill_mx_t4096", "layer_decode_mx_t64", "layer_prefill_a8w4_t4096",
                                  "layer_decode_a8w4_t64", "layer_prefill_a4w4_t4096", "layer_decode_a4w4_t64"])
def test_layer_mx_full_size_sampled_tokens(name):
    """The bench's workloads through moe_layer_forward_mx; y of a sample of
    tokens against the oracle run on those tokens alone (a token's output
    depends only on its own row and the weights)."""
    import moe_routed_expert_gb300 as M
    wl = WORKLOADS[name]
    inp = layer_inputs(wl, with_weights=False)
    wts = mx_layer_weights(wl)
    wf = wl.w_mx or wl.mx
    wsp = M.Workspace(M.moe_layer_mx_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.k))
    y = M.moe_layer_forward_mx(dev_bf16(inp["x"]), dev(inp["topk_ids"]), dev(inp["topk_w"]),
                               w_dev(wts["w1_q"], wf), dev(wts["w1_s"]), w_dev(wts["w2_q"], wf), dev(wts["w2_s"]),
                               x_fmt=wl.mx, w_fmt=wf, ws=wsp)
    assert M.read_status(wsp) == 0
    rng = np.random.default_rng(7)
    toks = np.sort(rng.choice(wl.T, size=min(8, wl.T), replace=False))
    ids = inp["topk_ids"][toks]
    used = np.unique(ids)
    remap = np.full(wl.E, -1, np.int32)
    remap[used] = np.arange(len(used))
    sub = lambda a: np.ascontiguousarray(a[used])
    y_want, _ = X.mx_layer_forward(f64(inp["x"][toks]), remap[ids], inp["topk_w"][toks], sub(wts["w1_q"]),
                                   sub(wts["w1_s"]), sub(wts["w2_q"]), sub(wts["w2_s"]), wl.mx, wf)
    assert_close("y", host_f64(y)[toks], y_want)


@pytest.mark.parametrize("xf,wf", [("e4m3", "e4m3"), ("e2m1", "e2m1")])
def test_gmm_forward_mx_sparse_batch_with_a_big_group(xf, wf):
    import torch
    import moe_routed_expert_gb300 as M
    rng = np.random.default_rng(53)
    counts = SPARSE_BIG_GROUP
    E, K, I = len(counts), 256, 256
    xq, xs, wq, ws, gl, _ = mx_gmm_case(rng, E, K, 2 * I, counts, xf, wf)
    wsp = M.Workspace(256)
    y = M.gmm_forward_mx(w_dev(xq, xf), dev(xs), w_dev(wq, wf), dev(ws), dev(gl), x_fmt=xf, w_fmt=wf, ws=wsp)
    assert M.read_status(wsp) == 0
    assert_close("y", y, X.mx_gmm(xq, xs, wq, ws, gl, xf, wf))
    h = torch.empty(int(sum(counts)), 2 * I, dtype=torch.bfloat16, device="cuda")
    aq, as_ = M.gmm_forward_mx(w_dev(xq, xf), dev(xs), w_dev(wq, wf), dev(ws), dev(gl), x_fmt=xf, w_fmt=wf,
                               activation=("swiglu", [7.0]), h_save=h, ws=wsp)
    assert M.read_status(wsp) == 0
    assert_close("h", h, X.mx_gmm(xq, xs, wq, ws, gl, xf, wf))
    check_act_codes(np_u8(aq), np_u8(as_), host_f64(h), O.activation("swiglu", [7.0]), X.activation_format(xf))


@pytest.mark.parametrize("xf,wf", [("e4m3", "e4m3"), ("e4m3", "e2m1")])
def test_gmm_forward_mx_max_experts(xf, wf):
    """1024 experts (the library's limit), most of them empty."""
    import moe_routed_expert_gb300 as M
    rng = np.random.default_rng(54)
    E, K, N = 1024, 128, 256
    counts = rng.choice([0, 0, 0, 1, 2, 4], size=E).astype(np.int64)
    counts[700] = 200
    xq, xs, wq, ws, gl, _ = mx_gmm_case(rng, E, K, N, counts, xf, wf)
    wsp = M.Workspace(256)
    y = M.gmm_forward_mx(w_dev(xq, xf), dev(xs), w_dev(wq, wf), dev(ws), dev(gl), x_fmt=xf, w_fmt=wf, ws=wsp)
    assert M.read_status(wsp) == 0
    assert_close("y", y, X.mx_gmm(xq, xs, wq, ws, gl, xf, wf))
