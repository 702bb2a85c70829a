"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, never against the oracle's own formulas retyped.

* the GMM page's worked example (tests/golden/gmm_worked_example.json);
* textbook special cases (E=1 is a plain matmul, checked against a brute-force
  Python triple loop; identity weights; sigma(0)=1/2; the combine of a k=1,
  w=1 route with identity experts is the identity);
* brute force on tiny inputs (Python's stable ``sorted`` for the dispatch order);
* exact finite differences and adjoint identities for every gradient;
* torch's float32 -> bfloat16 cast for the rounding helper.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- bf16 rounding
def test_round_to_bf16_special_values():
    r = O.round_to_bf16
    assert r(1.0) == 1.0
    assert r(1 + 2.0 ** -8) == 1.0                       # tie -> even (1.0000000)
    assert r(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6          # tie -> even (1.0000010)
    assert r(1 + 2.0 ** -8 + 2.0 ** -30) == 1 + 2.0 ** -7  # just above the tie
    assert r(-(1 + 2.0 ** -8)) == -1.0
    assert r(2.0 ** -133) == 2.0 ** -133                  # smallest subnormal
    assert r(2.0 ** -134) == 0.0                          # tie between 0 and 2^-133 -> 0
    assert r(1.5 * 2.0 ** -134) == 2.0 ** -133
    assert r(255 * 2.0 ** 120) == 255 * 2.0 ** 120        # largest finite bf16
    assert r(255.4 * 2.0 ** 120) == 255 * 2.0 ** 120
    assert np.isinf(r(255.5 * 2.0 ** 120))                # rounds past the largest -> inf
    assert np.isnan(r(np.nan)) and r(np.inf) == np.inf
    assert math.copysign(1.0, float(r(-0.0))) == -1.0


def test_round_to_bf16_matches_torch_cast():
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e-39).astype(np.float32),    # float32 subnormals
        (rng.standard_normal(5000) * 1e37).astype(np.float32),
        rng.integers(-2 ** 31, 2 ** 31, 20000).astype(np.int32).view(np.float32),  # random bit patterns
    ])
    v = v[np.isfinite(v)]
    want = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_to_bf16(v.astype(np.float64))
    np.testing.assert_array_equal(got, want)
    bits = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(O.f64_to_bf16_bits(v.astype(np.float64)), bits)
    np.testing.assert_array_equal(O.bf16_bits_to_f64(bits), want)


# ---------------------------------------------------------------- dispatch / permute
def worked_example_ids():
    g = load_golden("gmm_worked_example.json")
    T = 4
    k = 2
    ids = np.full((T, k), -1, np.int32)
    fill = [0] * T
    for t, e in g["pairs"]:
        ti, ei = int(t[1:]), int(e[1:])
        ids[ti, fill[ti]] = ei
        fill[ti] += 1
    return g, ids


def test_worked_example_counts_offsets_buckets():
    g, ids = worked_example_ids()
    E = g["num_experts"]
    row_id_map, sorted_flat, counts, off = O.stable_counting_sort(ids, E)
    assert counts.tolist() == g["group_list"]
    assert [[int(off[e]), int(off[e + 1])] for e in range(E)] == g["row_ranges"]
    k = ids.shape[1]
    for e in range(E):
        toks = ["t%d" % (f // k) for f in sorted_flat[off[e]:off[e + 1]]]
        assert toks == g["buckets"]["E%d" % e]
    # the histogram alone gives the page's group_list
    assert O.histogram(ids, E).tolist() == g["group_list"]


def test_dispatch_order_matches_brute_force_stable_sort():
    rng = np.random.default_rng(1)
    for trial in range(50):
        T, k, E = rng.integers(1, 12), rng.integers(1, 5), rng.integers(1, 7)
        ids = rng.integers(-1, E, size=(T, k)).astype(np.int32)
        row_id_map, sorted_flat, counts, off = O.stable_counting_sort(ids, E)
        flat = ids.ravel()
        want = [f for (_, f) in sorted((int(e), f) for f, e in enumerate(flat) if e >= 0)]
        assert sorted_flat.tolist() == want
        assert int(counts.sum()) == int((flat >= 0).sum())
        for f, e in enumerate(flat):
            if e < 0:
                assert row_id_map[f] == -1
            else:
                assert sorted_flat[row_id_map[f]] == f
                assert off[e] <= row_id_map[f] < off[e + 1]
        assert np.all(np.diff(off) >= 0)


def test_empty_group_leaves_later_offsets_intact():
    rng = np.random.default_rng(2)
    ids = rng.integers(0, 4, size=(9, 3)).astype(np.int32)
    _, _, counts, off = O.stable_counting_sort(ids, 4)
    # insert an empty expert at position 2: experts >= 2 shift up by one
    ids2 = np.where(ids >= 2, ids + 1, ids).astype(np.int32)
    _, _, counts2, off2 = O.stable_counting_sort(ids2, 5)
    assert counts2[2] == 0
    assert off2[2] == off2[3]
    assert off2.tolist() == off[:3].tolist() + off[2:].tolist()


def test_permute_rows_are_token_copies_and_bad_ids_raise():
    rng = np.random.default_rng(3)
    T, k, E, H = 7, 3, 5, 4
    ids = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    x = rng.standard_normal((T, H))
    x_perm, counts, row_id_map, sorted_flat = O.moe_permute(x, ids, E)
    for f in range(T * k):
        if row_id_map[f] >= 0:
            np.testing.assert_array_equal(x_perm[row_id_map[f]], x[f // k])
    with pytest.raises(ValueError):
        O.moe_permute(x, np.full((T, k), E, np.int32), E)
    with pytest.raises(ValueError):
        O.moe_permute(x, np.full((T, k), -2, np.int32), E)


# ---------------------------------------------------------------- grouped matmul
def brute_matmul(a, b):
    n, m, p = len(a), len(b), len(b[0])
    return [[sum(a[i][l] * b[l][j] for l in range(m)) for j in range(p)] for i in range(n)]


def test_gmm_single_group_is_plain_matmul():
    rng = np.random.default_rng(4)
    M, K, N = 6, 5, 3
    x = rng.standard_normal((M, K))
    w = rng.standard_normal((1, K, N))
    y = O.gmm_forward(x, w, [M], store=None)
    np.testing.assert_allclose(y, np.array(brute_matmul(x.tolist(), w[0].tolist())), rtol=0, atol=1e-12)


def test_gmm_row_to_weight_map_of_the_worked_example():
    g = load_golden("gmm_worked_example.json")
    gl = g["group_list"]
    K = N = 3
    w = np.stack([(e + 1) * np.eye(K) for e in range(4)])
    x = np.arange(1, 1 + sum(gl) * K, dtype=np.float64).reshape(-1, K)
    y = O.gmm_forward(x, w, gl, store=None)
    for e, (s, t) in enumerate(g["row_ranges"]):
        np.testing.assert_array_equal(y[s:t], (e + 1) * x[s:t])
    # identity weights: Y = X exactly, also after bf16 storage of bf16 inputs
    xb = O.round_to_bf16(np.random.default_rng(5).standard_normal((5, K)))
    np.testing.assert_array_equal(O.gmm_forward(xb, np.stack([np.eye(K)] * 4), gl), xb)
    with pytest.raises(ValueError):
        O.gmm_forward(x, w, [1, 2, 0, 1])


def test_gmm_expert_relabel_permutes_blocks():
    rng = np.random.default_rng(6)
    gl = np.array([3, 0, 2, 4])
    K, N = 4, 6
    x = rng.standard_normal((gl.sum(), K))
    w = rng.standard_normal((4, K, N))
    y = O.gmm_forward(x, w, gl, store=None)
    perm = np.array([2, 0, 3, 1])
    off = np.concatenate([[0], np.cumsum(gl)])
    xb = np.concatenate([x[off[p]:off[p + 1]] for p in perm])
    yb = np.concatenate([y[off[p]:off[p + 1]] for p in perm])
    np.testing.assert_allclose(O.gmm_forward(xb, w[perm], gl[perm], store=None), yb, atol=1e-12)


def test_gmm_backward_finite_differences_and_adjoint():
    rng = np.random.default_rng(7)
    gl = [4, 0, 3]
    M, K, N = 7, 5, 3        # K != N so a transposed operand cannot pass
    x = rng.standard_normal((M, K))
    w = rng.standard_normal((3, K, N))
    gy = rng.standard_normal((M, N))
    dx, dw = O.gmm_backward(x, w, gl, gy, store=None)

    def L(xx, ww):
        return float(np.sum(gy * O.gmm_forward(xx, ww, gl, store=None)))

    eps = 1e-3  # L is linear in each argument, so the central difference is exact up to rounding
    for i in range(M):
        for j in range(K):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += eps
            xm[i, j] -= eps
            assert abs((L(xp, w) - L(xm, w)) / (2 * eps) - dx[i, j]) < 1e-9
    for e in range(3):
        for i in range(K):
            for j in range(N):
                wp, wm = w.copy(), w.copy()
                wp[e, i, j] += eps
                wm[e, i, j] -= eps
                assert abs((L(x, wp) - L(x, wm)) / (2 * eps) - dw[e, i, j]) < 1e-9
    assert np.all(dw[1] == 0)  # empty group
    y = O.gmm_forward(x, w, gl, store=None)
    lhs = np.sum(gy * y)
    assert abs(lhs - np.sum(dx * x)) < 1e-9 and abs(lhs - np.sum(dw * w)) < 1e-9


# ---------------------------------------------------------------- SwiGLU
def test_sigmoid_silu_textbook_values():
    assert O.sigmoid(0.0) == 0.5
    assert O.silu(0.0) == 0.0
    assert abs(O.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(O.silu(40.0) - 40.0) < 1e-12
    assert abs(O.silu(-40.0)) < 1e-12
    assert O.silu(-1000.0) == 0.0 or abs(O.silu(-1000.0)) < 1e-300


def test_swiglu_gate_first_and_clip():
    s = lambda z: 1.0 / (1.0 + math.exp(-z))
    h = np.array([[1.0, -2.0, 2.0, 0.5]])   # G = [1, -2], U = [2, 0.5]
    a = O.swiglu(h, None, store=None)
    np.testing.assert_allclose(a, [[1.0 * s(1.0) * 2.0, -2.0 * s(-2.0) * 0.5]], rtol=1e-15)
    # c = 7: G = 10 -> 7, U = 10 -> 7, U = -10 -> -7
    h = np.array([[10.0, 10.0, 3.0, -10.0]])
    a = O.swiglu(h, 7.0, store=None)
    np.testing.assert_allclose(a, [[7 * s(7) * 3.0, 7 * s(7) * -7.0]], rtol=1e-15)
    # only the gate is clipped from above: a very negative G is kept
    a = O.swiglu(np.array([[-10.0, 1.0]]), 7.0, store=None)
    assert abs(a[0, 0] - (-10 * s(-10))) < 1e-15
    # c = 0 and c unset both mean no clip
    h = np.random.default_rng(8).standard_normal((5, 8)) * 20
    np.testing.assert_array_equal(O.swiglu(h, 0.0, store=None), O.swiglu(h, None, store=None))
    with pytest.raises(ValueError):
        O.swiglu(h, -1.0)


def test_swiglu_backward_finite_differences():
    rng = np.random.default_rng(9)
    for clip in (None, 1.5):
        h = rng.standard_normal((6, 10)) * 2
        h[np.abs(np.abs(h) - 1.5) < 1e-2] += 0.1   # stay off the clip kinks
        da = rng.standard_normal((6, 5))
        dh = O.swiglu_backward(h, da, clip, store=None)
        eps = 1e-6
        for i in range(6):
            for j in range(10):
                hp, hm = h.copy(), h.copy()
                hp[i, j] += eps
                hm[i, j] -= eps
                fd = (np.sum(da * O.swiglu(hp, clip, store=None)) - np.sum(da * O.swiglu(hm, clip, store=None))) / (2 * eps)
                assert abs(fd - dh[i, j]) < 1e-7 * max(1.0, abs(fd))


# ---------------------------------------------------------------- activation variants ([MegaMoE])
def test_activation_parameters_and_defaults():
    # the empty-list defaults the pages state: no clip, alpha 1.702, beta 1.0, no linear_beta
    a = O.activation("swigluoai")
    assert (a["c"], a["alpha"], a["beta"]) == (np.inf, 1.702, 1.0)
    a = O.activation("situglu")
    assert (a["beta"], a["linear_beta"]) == (1.0, None)
    assert O.activation("swiglustep", [0.0])["c"] == np.inf          # clamp 0: no clip
    assert O.activation("swigluoai", [5.0, 2.0, -0.5])["alpha"] == 2.0
    assert O.activation("situglu", [2.0, 3.0])["linear_beta"] == 3.0
    for kind, params in (("swiglu", [1.0, 2.0]), ("swigluoai", [1.0]), ("situglu", [1.0, 2.0, 3.0]),
                         ("situglu", [0.0]), ("situglu", [1.0, -1.0]), ("gelu", [])):
        with pytest.raises(ValueError):
            O.activation(kind, params)


def test_activation_variants_reduce_to_swiglu():
    h = np.random.default_rng(21).standard_normal((6, 16)) * 3
    for clip in (None, 1.5):
        sw = O.swiglu(h, clip, store=None)
        np.testing.assert_array_equal(O.gated_activation(h, O.activation("swiglu", [clip or 0.0]), store=None), sw)
        # swigluoai with alpha = 1 and beta = 0 is G_c sigma(G_c) U_c
        oai = O.gated_activation(h, O.activation("swigluoai", [clip or 0.0, 1.0, 0.0]), store=None)
        np.testing.assert_allclose(oai, sw, rtol=1e-14, atol=1e-15)
    # swiglustep without a clip is SiLU(G) U
    np.testing.assert_allclose(O.gated_activation(h, O.activation("swiglustep"), store=None),
                               O.swiglu(h, None, store=None), rtol=1e-14, atol=1e-15)
    # situglu: beta tanh(G / beta) -> G as beta grows, and so does linear_beta tanh(U / linear_beta) -> U
    big = O.gated_activation(h, O.activation("situglu", [1e6, 1e6]), store=None)
    np.testing.assert_allclose(big, O.swiglu(h, None, store=None), rtol=1e-9, atol=1e-12)
    big = O.gated_activation(h, O.activation("situglu", [1e6]), store=None)
    np.testing.assert_allclose(big, O.swiglu(h, None, store=None), rtol=1e-9, atol=1e-12)


def test_activation_variants_by_hand():
    s = lambda z: 1.0 / (1.0 + math.exp(-z))
    # swiglustep: SiLU(20) > c = 5 is cut to 5; U = 3 is inside the clip
    a = O.gated_activation(np.array([[20.0, 3.0]]), O.activation("swiglustep", [5.0]), store=None)
    assert abs(a[0, 0] - 15.0) < 1e-12
    # ... while the gate itself is not clipped: G = -3 keeps SiLU(-3); U = 9 -> 5
    a = O.gated_activation(np.array([[-3.0, 9.0]]), O.activation("swiglustep", [5.0]), store=None)
    assert abs(a[0, 0] - (-3.0 * s(-3.0) * 5.0)) < 1e-12
    # swigluoai at G = 0 is 0 whatever U; with G = c = 2, alpha = 1.702, U = 10 -> 2, beta = 1
    oai = O.activation("swigluoai", [2.0, 1.702, 1.0])
    assert O.gated_activation(np.array([[0.0, 5.0]]), oai, store=None)[0, 0] == 0.0
    a = O.gated_activation(np.array([[4.0, 10.0]]), oai, store=None)
    assert abs(a[0, 0] - 2.0 * s(1.702 * 2.0) * 3.0) < 1e-12
    # situglu with beta = 1 at G = 1: tanh(1) sigma(1) U
    a = O.gated_activation(np.array([[1.0, 2.0]]), O.activation("situglu", [1.0]), store=None)
    assert abs(a[0, 0] - math.tanh(1.0) * s(1.0) * 2.0) < 1e-12
    # situglu's L: U = linear_beta * artanh(1/2) gives L = linear_beta / 2
    lb = 3.0
    a = O.gated_activation(np.array([[1.0, lb * math.atanh(0.5)]]), O.activation("situglu", [1.0, lb]), store=None)
    assert abs(a[0, 0] - math.tanh(1.0) * s(1.0) * lb / 2) < 1e-12
    # gradients at G = 0 by hand: swigluoai d/dG = sigma(0) (U + beta); situglu d/dG = sigma(0) L(U)
    d = O.gated_activation_backward(np.array([[0.0, 1.0]]), np.array([[1.0]]), O.activation("swigluoai"), store=None)
    assert abs(d[0, 0] - 0.5 * 2.0) < 1e-12 and d[0, 1] == 0.0
    d = O.gated_activation_backward(np.array([[0.0, 2.0]]), np.array([[1.0]]), O.activation("situglu"), store=None)
    assert abs(d[0, 0] - 0.5 * 2.0) < 1e-12 and d[0, 1] == 0.0


@pytest.mark.parametrize("kind,params", [("swiglu", [1.5]), ("swiglustep", [0.6]), ("swigluoai", [1.5, 1.702, 1.0]),
                                         ("swigluoai", []), ("situglu", [0.7]), ("situglu", [1.3, 0.8])])
def test_activation_variants_backward_finite_differences(kind, params):
    act = O.activation(kind, params)
    rng = np.random.default_rng(22)
    h = rng.standard_normal((5, 12)) * 2
    I = 6
    c = act["c"]
    if np.isfinite(c):  # stay off the kinks
        h[np.abs(np.abs(h) - c) < 2e-2] += 0.1
        if kind == "swiglustep":
            g = h[:, :I]
            near = np.abs(O.silu(g) - c) < 2e-2
            g[near] += 0.2
    da = rng.standard_normal((5, I))
    dh = O.gated_activation_backward(h, da, act, store=None)
    eps = 1e-6
    for i in range(5):
        for j in range(12):
            hp, hm = h.copy(), h.copy()
            hp[i, j] += eps
            hm[i, j] -= eps
            fd = (np.sum(da * O.gated_activation(hp, act, store=None)) -
                  np.sum(da * O.gated_activation(hm, act, store=None))) / (2 * eps)
            assert abs(fd - dh[i, j]) < 1e-7 * max(1.0, abs(fd)), (kind, i, j, fd, dh[i, j])


# ---------------------------------------------------------------- combine and its gradients
def test_combine_identity_route_returns_input():
    rng = np.random.default_rng(10)
    T, H, E = 9, 6, 4
    ids = rng.integers(0, E, size=(T, 1)).astype(np.int32)
    x = rng.standard_normal((T, H))
    x_perm, counts, rmap, _ = O.moe_permute(x, ids, E)
    y_perm = O.gmm_forward(x_perm, np.stack([np.eye(H)] * E), counts, store=None)
    y = O.moe_unpermute(y_perm, rmap, np.ones((T, 1)), T, 1, store=None)
    np.testing.assert_array_equal(y, x)


def test_combine_worked_example_by_hand():
    g, ids = worked_example_ids()
    T, k = ids.shape
    rmap, sorted_flat, counts, off = O.stable_counting_sort(ids, g["num_experts"])
    # rows: E0:[t2] -> 0, E1:[t0,t1] -> 1,2, E3:[t0,t3] -> 3,4
    assert rmap.tolist() == [1, 3, 2, -1, 0, -1, 4, -1]
    y_perm = np.array([[1.0], [10.0], [100.0], [1000.0], [10000.0]])
    w = np.array([[0.25, 0.75], [1.0, 9.0], [1.0, 9.0], [0.5, 9.0]])
    y = O.moe_unpermute(y_perm, rmap, w, T, k, store=None)
    np.testing.assert_allclose(y.ravel(), [0.25 * 10 + 0.75 * 1000, 100.0, 1.0, 0.5 * 10000])
    dx = O.moe_permute_backward(y_perm, rmap, T, k, store=None)
    np.testing.assert_allclose(dx.ravel(), [10 + 1000, 100.0, 1.0, 10000.0])


def test_combine_backward_finite_differences():
    rng = np.random.default_rng(11)
    T, k, E, H = 5, 3, 4, 6
    ids = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    _, counts, rmap, _ = O.moe_permute(np.zeros((T, H)), ids, E)
    R = int(counts.sum())
    y_perm = rng.standard_normal((R, H))
    w = rng.standard_normal((T, k))
    gy = rng.standard_normal((T, H))
    dyp, dpr = O.moe_unpermute_backward(gy, y_perm, rmap, w, T, k, store=None)
    L = lambda yp, ww: float(np.sum(gy * O.moe_unpermute(yp, rmap, ww, T, k, store=None)))
    eps = 1e-3
    for r in range(R):
        for h in range(H):
            p, m = y_perm.copy(), y_perm.copy()
            p[r, h] += eps
            m[r, h] -= eps
            assert abs((L(p, w) - L(m, w)) / (2 * eps) - dyp[r, h]) < 1e-9
    for t in range(T):
        for j in range(k):
            p, m = w.copy(), w.copy()
            p[t, j] += eps
            m[t, j] -= eps
            assert abs((L(y_perm, p) - L(y_perm, m)) / (2 * eps) - dpr[t, j]) < 1e-9
            if rmap[t * k + j] < 0:
                assert dpr[t, j] == 0.0


def test_token_grad_is_adjoint_of_permute():
    rng = np.random.default_rng(12)
    T, k, E, H = 8, 3, 5, 4
    ids = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    x = rng.standard_normal((T, H))
    x_perm, counts, rmap, _ = O.moe_permute(x, ids, E)
    gp = rng.standard_normal(x_perm.shape)
    dx = O.moe_permute_backward(gp, rmap, T, k, store=None)
    assert abs(np.sum(dx * x) - np.sum(gp * x_perm)) < 1e-10


# ---------------------------------------------------------------- whole layer
def test_layer_single_expert_is_dense_swiglu_mlp():
    rng = np.random.default_rng(13)
    T, H, I = 6, 8, 4
    x = rng.standard_normal((T, H))
    w1 = rng.standard_normal((1, H, 2 * I))
    w2 = rng.standard_normal((1, I, H))
    y, _ = O.moe_layer_forward(x, np.zeros((T, 1), np.int32), np.ones((T, 1)), w1, w2, None, store=None)
    gate, up = x @ w1[0][:, :I], x @ w1[0][:, I:]
    want = (gate / (1 + np.exp(-gate)) * up) @ w2[0]
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("clip", [None, 0.8])
def test_layer_backward_finite_differences(clip):
    rng = np.random.default_rng(14)
    T, H, I, E, k = 5, 6, 3, 4, 2
    ids = np.array([[0, 2], [2, -1], [3, 0], [0, 3], [2, 0]], np.int32)   # expert 1 empty
    x = rng.standard_normal((T, H))
    tw = rng.random((T, k))
    w1 = rng.standard_normal((E, H, 2 * I)) * 0.5
    w2 = rng.standard_normal((E, I, H)) * 0.5
    gy = rng.standard_normal((T, H))
    y, saved = O.moe_layer_forward(x, ids, tw, w1, w2, clip, store=None)
    if clip is not None:  # keep every pre-activation off the clip kinks
        hh = saved["h"]
        assert np.min(np.abs(np.abs(hh) - clip)) > 1e-3
    dx, dw1, dw2, dpr = O.moe_layer_backward(gy, saved, tw, w1, w2, clip, store=None)

    def L(xx=x, t=tw, a=w1, b=w2):
        return float(np.sum(gy * O.moe_layer_forward(xx, ids, t, a, b, clip, store=None)[0]))

    eps = 1e-6

    def fd(arr, idx, **kw):
        p, m = arr.copy(), arr.copy()
        p[idx] += eps
        m[idx] -= eps
        return (L(**{kw["name"]: p}) - L(**{kw["name"]: m})) / (2 * eps)

    for name, arr, grad in (("xx", x, dx), ("t", tw, dpr), ("a", w1, dw1), ("b", w2, dw2)):
        for idx in np.ndindex(arr.shape):
            g = fd(arr, idx, name=name)
            assert abs(g - grad[idx]) < 1e-6 * max(1.0, abs(g)), (name, idx, g, grad[idx])
    assert np.all(dw1[1] == 0) and np.all(dw2[1] == 0)
    assert dpr[1, 1] == 0.0
