"""Pins of the MX oracle (oracle/mx_oracle.py: MXFP8, and MXFP4 weights) to
things other than itself.

- The fp8 element formats: every code's value against torch's own float8
  dtypes (a library decode), and the format constants the pages' type names
  fix (largest finite value, smallest subnormal, 1.0, NaN / infinity codes).
- Rounding: against torch's float8 conversion (nearest, ties to even) wherever
  it does not saturate, exact midpoints, and the saturation that reading M2
  adds on top.
- Q_MX: hand-computed groups ("MegaMoE", A8W8-FP 量化场景: group of 32, shared
  exponent, E8M0 scale), the error bound that follows from the element
  format, and that dequantising returns exactly representable inputs.
- The MX grouped matmul against a torch float64 matmul of torch-dequantised
  operands, and the MX layer against a per-token evaluation of the four stages
  that takes no permute at all.
- A4W4-FP: the per-token layer pin with E2M1 tokens and an E4M3 activation.
- FLOAT4_E2M1 ("MegaMoE", A8W4-FP 量化场景): the 16 codes against the type's
  eight magnitudes, ties to the even code, saturation at 6, hand-computed Q_MX
  groups, and the same error bound, exactness, GMM and per-token layer pins
  with the weights decoded from that value table.
"""
import numpy as np
import pytest
import torch

import oracle as O
from oracle import mx_oracle as X

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

TORCH_FP8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
# FLOAT4_E2M1's eight magnitudes (the type's definition: no infinities, no NaN)
E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def torch_decode(codes, fmt):
    t = torch.from_numpy(np.asarray(codes, dtype=np.uint8).copy())
    return t.view(TORCH_FP8[fmt]).to(torch.float64).numpy()


def torch_encode(v, fmt):
    return torch.from_numpy(np.asarray(v, np.float64)).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_decode_matches_torch_for_every_code(fmt):
    codes = np.arange(256)
    got = X.fp8_decode(codes, fmt)
    want = torch_decode(codes, fmt)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))


def test_fp8_format_constants():
    d4 = lambda c: float(X.fp8_decode([c], "e4m3")[0])
    d5 = lambda c: float(X.fp8_decode([c], "e5m2")[0])
    assert d4(0x38) == 1.0 and d4(0x7E) == 448.0 and d4(0x01) == 2.0 ** -9 and np.isnan(d4(0x7F))
    assert d4(0x08) == 2.0 ** -6   # smallest normal
    assert d5(0x3C) == 1.0 and d5(0x7B) == 57344.0 and d5(0x01) == 2.0 ** -16 and d5(0x7C) == np.inf
    assert np.isnan(d5(0x7D)) and d5(0xFC) == -np.inf
    assert X.FP8_FORMATS["e4m3"]["emax"] == 8 and 2.0 ** 8 <= 448 < 2.0 ** 9
    assert X.FP8_FORMATS["e5m2"]["emax"] == 15 and 2.0 ** 15 <= 57344 < 2.0 ** 16
    assert X.e8m0_decode([127])[0] == 1.0 and X.e8m0_decode([0])[0] == 2.0 ** -127
    assert X.e8m0_decode([254])[0] == 2.0 ** 127 and np.isnan(X.e8m0_decode([255])[0])


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_encode_matches_torch_in_range(fmt):
    rng = np.random.default_rng(7)
    mx = X.FP8_FORMATS[fmt]["max"]
    codes, vals = X.fp8_finite_values(fmt)
    mids = (vals[1:] + vals[:-1]) / 2                      # exact ties
    v = np.concatenate([
        rng.uniform(-mx, mx, 20000),
        np.exp2(rng.uniform(-20, np.log2(mx), 20000)) * rng.choice([-1, 1], 20000),
        mids, -mids, vals, -vals, [0.0, -0.0],
    ])
    assert np.array_equal(X.fp8_encode(v, fmt), torch_encode(v, fmt))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_encode_saturates_and_round_trips(fmt):
    f = X.FP8_FORMATS[fmt]
    big = np.array([f["max"] * 1.01, f["max"] * 1.5, 1e30, np.inf])
    assert np.all(X.fp8_encode(big, fmt) == X.fp8_encode([f["max"]], fmt)[0])
    assert np.all(X.fp8_encode(-big, fmt) == (X.fp8_encode([f["max"]], fmt)[0] | 0x80))
    assert X.fp8_encode([np.nan], fmt)[0] == f["nan_code"]
    codes = np.arange(256)
    vals = X.fp8_decode(codes, fmt)
    fin = np.isfinite(vals)
    assert np.array_equal(X.fp8_encode(vals[fin], fmt), codes[fin])


def test_mx_quantize_hand_groups_e4m3():
    g = np.zeros((7, 32))
    g[0, 0] = 1.0            # amax 1: X = 2^(0-8); 1 * 2^8 = 256 -> 0x78
    g[1, :2] = [1.75, -0.5]  # 1.75 * 256 = 448 -> 0x7E; -128 -> 0xF0
    g[2, 0] = 1.9            # 486.4 saturates to 448
    g[3, 5] = -0.0           # all zero: scale code 0, signed zeros kept
    g[4, 3] = 2.0 ** 100     # scale 2^92 -> code 219
    g[5, 0] = 2.0 ** -140    # exponent clamps at -127: 2^-13 rounds to 0
    g[6, :3] = [3.0, 0.1, np.nan]
    q, s = X.mx_quantize(g, "e4m3")
    assert s.tolist() == [[119], [119], [119], [0], [219], [0], [255]]
    assert q[0, 0] == 0x78 and q[1, 0] == 0x7E and q[1, 1] == 0xF0 and q[2, 0] == 0x7E
    assert q[3, 5] == 0x80 and q[3, 0] == 0x00
    assert q[4, 3] == 0x78 and q[5, 0] == 0
    assert np.all(q[6] == 0x7F)


def test_mx_quantize_hand_groups_e5m2():
    g = np.zeros((2, 32))
    g[0, :2] = [1.0, 0.75]   # X = 2^(0-15): 2^15 -> 0x78; 0.75 * 2^15 = 1.5 * 2^14 -> 0x76
    g[1, 0] = 1.9            # 1.9 * 2^15 = 62259 saturates to 57344 (0x7B)
    q, s = X.mx_quantize(g, "e5m2")
    assert s.tolist() == [[112], [112]]
    assert q[0, 0] == 0x78 and q[0, 1] == 0x76 and q[1, 0] == 0x7B


def test_e2m1_codes_values_and_rounding():
    codes = np.arange(16)
    assert X.fp8_decode(codes, "e2m1").tolist() == E2M1_VALUES + [-v for v in E2M1_VALUES]
    assert X.FP8_FORMATS["e2m1"]["emax"] == 2 and 2.0 ** 2 <= 6.0 < 2.0 ** 3
    # ties go to the even code; beyond 6 saturates; signed zero and NaN per the readings
    v = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 1e9, -0.0, -1.5, np.nan, 0.26, 5.01]
    want = [0, 2, 2, 4, 4, 6, 6, 7, 7, 8, 11, 7, 1, 7]
    assert X.fp8_encode(v, "e2m1").tolist() == want
    vals = X.fp8_decode(codes, "e2m1")
    assert np.array_equal(X.fp8_encode(vals, "e2m1"), codes)
    g = np.zeros((3, 32))
    g[0, :2] = [1.0, 0.3]      # X = 2^(0-2): 4 -> code 6, 1.2 -> 1.0 (code 2)
    g[1, 0] = 1.5              # 6 -> code 7
    g[2, :2] = [1.9, -0.1]     # 7.6 saturates to 6; -0.4 -> -0.5 (code 9)
    q, sc = X.mx_quantize(g, "e2m1")
    assert sc.tolist() == [[125], [125], [125]]
    assert q[0, :2].tolist() == [6, 2] and q[1, 0] == 7 and q[2, :2].tolist() == [7, 9]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "e2m1"])
def test_mx_quantize_error_bound(fmt):
    """Each element lies within half a step of its dequantised value, the step
    being that of the element format's binade of |x| / X (or the subnormal step
    below the smallest normal); saturated elements lie in [max X, 2^(emax+1) X)."""
    f = X.FP8_FORMATS[fmt]
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 256)) * np.exp2(rng.integers(-30, 30, (64, 1)))
    q, s = X.mx_quantize(x, fmt)
    dq = X.mx_dequantize(q, s, fmt)
    scale = np.repeat(X.e8m0_decode(s), 32, axis=1)
    r = np.abs(x) / scale
    assert np.all(r < 2.0 ** (f["emax"] + 1))
    assert np.all(np.max(r.reshape(64, -1, 32), axis=2) >= 2.0 ** f["emax"])
    binade = np.maximum(np.floor(np.log2(np.maximum(r, 1e-300))), 1 - f["bias"])
    step = np.exp2(binade - f["mbits"]) * scale
    sat = r > f["max"]
    err = np.abs(dq - x)
    assert np.all(err[~sat] <= step[~sat] / 2)
    assert np.all(np.abs(dq[sat]) == f["max"] * scale[sat])


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "e2m1"])
def test_mx_quantize_is_exact_on_representable_groups(fmt):
    rng = np.random.default_rng(11)
    codes, vals = X.fp8_finite_values(fmt)
    v = rng.choice(vals, (16, 128)) * rng.choice([-1, 1], (16, 128))
    v[:, ::32] = vals[-1]                                    # amax = max finite in every group
    x = v * np.exp2(rng.integers(-20, 20, (16, 1)))
    q, s = X.mx_quantize(x, fmt)
    assert np.array_equal(X.mx_dequantize(q, s, fmt), x)


def _torch_dequant(q, s, fmt):
    """Dequantise with an independent element decode: torch's float8 dtypes, or
    the E2M1 value table."""
    if fmt == "e2m1":
        c = np.asarray(q, np.int64)
        v = np.array(E2M1_VALUES)[c & 7] * np.where(c & 8, -1.0, 1.0)
    else:
        v = torch_decode(q, fmt)
    sc = np.exp2(np.asarray(s, np.float64) - 127)
    return (v.reshape(v.shape[:-1] + (-1, 32)) * sc[..., None]).reshape(v.shape)


def test_mx_gmm_with_e2m1_weights():
    rng = np.random.default_rng(6)
    E, K, N = 2, 128, 32
    counts = np.array([7, 4])
    xq = rng.integers(0, 256, (11, K)).astype(np.uint8)
    xq[(xq & 0x7F) == 0x7F] = 0x11
    wq = rng.integers(0, 16, (E, N, K)).astype(np.uint8)
    xs = rng.integers(115, 130, (11, K // 32)).astype(np.uint8)
    ws = rng.integers(115, 130, (E, N, K // 32)).astype(np.uint8)
    got = X.mx_gmm(xq, xs, wq, ws, counts, "e4m3", "e2m1", store=None)
    xd = _torch_dequant(xq, xs, "e4m3")
    wd = _torch_dequant(wq, ws, "e2m1")
    want = np.concatenate([xd[:7] @ wd[0].T, xd[7:] @ wd[1].T])
    assert np.allclose(got, want, rtol=1e-12, atol=0)


def test_mx_gmm_against_torch_dequant_matmul():
    rng = np.random.default_rng(5)
    E, K, N = 3, 128, 64
    counts = np.array([5, 0, 9])
    M = counts.sum()
    xq = rng.integers(0, 256, (M, K)).astype(np.uint8)
    xq[(xq & 0x7F) == 0x7F] = 0x11                            # no NaN codes
    wq = rng.integers(0, 256, (E, N, K)).astype(np.uint8)
    wq[(wq & 0x7F) >= 0x7C] = 0x22                            # no e5m2 inf / NaN
    xs = rng.integers(110, 135, (M, K // 32)).astype(np.uint8)
    ws = rng.integers(110, 135, (E, N, K // 32)).astype(np.uint8)
    got = X.mx_gmm(xq, xs, wq, ws, counts, "e4m3", "e5m2", store=None)
    xd = torch.from_numpy(_torch_dequant(xq, xs, "e4m3"))
    wd = torch.from_numpy(_torch_dequant(wq, ws, "e5m2"))
    off = np.concatenate([[0], np.cumsum(counts)])
    for g in range(E):
        want = (xd[off[g]:off[g + 1]] @ wd[g].T).numpy()
        assert np.allclose(got[off[g]:off[g + 1]], want, rtol=1e-12, atol=0)


# (token type, weight type, activation type): A8W8-FP, A8W4-FP, A4W4-FP, whose
# activation is E4M3 although its tokens are E2M1 ("MegaMoE", A4W4-FP 量化场景)
LAYER_FORMATS = [("e4m3", "e4m3", "e4m3"), ("e5m2", "e5m2", "e5m2"), ("e4m3", "e2m1", "e4m3"),
                 ("e2m1", "e2m1", "e4m3")]


@pytest.mark.parametrize("x_fmt,w_fmt,a_fmt", LAYER_FORMATS)
def test_mx_layer_matches_per_token_stages(x_fmt, w_fmt, a_fmt):
    """Stage by stage for each token on its own: quantise the token's row, the
    gate_up product with expert e's weights, bf16, the activation, quantise,
    the down product, bf16, then the weighted sum over its k slots."""
    rng = np.random.default_rng(9)
    T, H, I, E, k = 6, 128, 128, 4, 2
    x = O.round_to_bf16(rng.standard_normal((T, H)))
    ids = np.array([[0, 2], [2, 3], [1, 0], [3, 2], [0, -1], [2, 1]], np.int32)
    tw = rng.uniform(0.1, 1.0, (T, k)).astype(np.float32)
    w1 = rng.standard_normal((E, 2 * I, H)) / np.sqrt(H)
    w2 = rng.standard_normal((E, H, I)) / np.sqrt(I)
    w1q, w1s = X.mx_quantize(w1, w_fmt)
    w2q, w2s = X.mx_quantize(w2, w_fmt)
    act = O.activation("swiglu", [7.0])
    y, saved = X.mx_layer_forward(x, ids, tw, w1q, w1s, w2q, w2s, x_fmt, w_fmt, act)
    w1d = _torch_dequant(w1q, w1s, w_fmt)
    w2d = _torch_dequant(w2q, w2s, w_fmt)
    want = np.zeros((T, H))
    for t in range(T):
        acc = np.zeros(H)
        for j in range(k):
            e = ids[t, j]
            if e < 0:
                continue
            xq, xs = X.mx_quantize(x[t:t + 1], x_fmt)
            xr = _torch_dequant(xq, xs, x_fmt)
            h = O.round_to_bf16(xr @ w1d[e].T)
            g, u = h[:, :I], h[:, I:]
            gc = np.minimum(g, 7.0)
            a = gc / (1 + np.exp(-gc)) * np.clip(u, -7.0, 7.0)
            aq, as_ = X.mx_quantize(a, a_fmt)
            o = O.round_to_bf16(_torch_dequant(aq, as_, a_fmt) @ w2d[e].T)
            acc += float(tw[t, j]) * o[0]
        want[t] = O.round_to_bf16(acc)
    assert np.array_equal(y, want)
    # the quantised activation holds codes of a_fmt: E2M1 codes stop at 15
    assert saved["aq"].max() > 15 or a_fmt == "e2m1"


def test_mx_layer_close_to_unquantised_layer():
    """Quantisation noise only: the MX layer stays within a few percent (RMS)
    of the bf16 layer evaluated on the same dequantised weights."""
    rng = np.random.default_rng(13)
    T, H, I, E, k = 32, 256, 128, 4, 2
    x = O.round_to_bf16(rng.standard_normal((T, H)))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    tw = rng.uniform(0.1, 1.0, (T, k)).astype(np.float32)
    w1q, w1s = X.mx_quantize(rng.standard_normal((E, 2 * I, H)) / np.sqrt(H), "e4m3")
    w2q, w2s = X.mx_quantize(rng.standard_normal((E, H, I)) / np.sqrt(I), "e4m3")
    y, _ = X.mx_layer_forward(x, ids, tw, w1q, w1s, w2q, w2s, "e4m3", "e4m3", None, store=None)
    w1 = np.transpose(X.mx_dequantize(w1q, w1s, "e4m3"), (0, 2, 1))
    w2 = np.transpose(X.mx_dequantize(w2q, w2s, "e4m3"), (0, 2, 1))
    ref, _ = O.moe_layer_forward(x, ids, tw, w1, w2, store=None)
    rel = np.sqrt(np.mean((y - ref) ** 2) / np.mean(ref ** 2))
    assert 1e-3 < rel < 0.08, rel
