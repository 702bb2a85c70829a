"""Parity of the tcgen05 grouped matmul (forward, SwiGLU epilogue, dX, dW)
with the oracle, elementwise within the pages' bf16 tolerance, over ragged
groups (empty groups, groups shorter than a tile, rows past the group sum),
sizes that span several tiles with partial edges, and the workload shapes."""
import numpy as np
import pytest

import oracle as O
from tests._util import assert_close, dev, dev_bf16, f64, host_f64
from workloads import WORKLOADS, gmm_inputs, normal_bf16

pytestmark = pytest.mark.gpu


def counts_with_empties(rng, E, M, n_empty):
    c = np.zeros(E, np.int64)
    live = rng.permutation(E)[n_empty:]
    cuts = np.sort(rng.integers(0, M + 1, size=len(live) - 1))
    c[live] = np.diff(np.concatenate([[0], cuts, [M]]))
    return c


def gpu_forward(x, w, gl, epilogue=0, clip=0.0, want_h=False):
    import torch
    import moe_routed_expert_gb300 as M
    ws = M.Workspace(256)
    xd, wd = dev_bf16(x), dev_bf16(w)
    h = torch.empty(x.shape[0], w.shape[2], dtype=torch.bfloat16, device="cuda") if want_h else None
    y = M.gmm_forward(xd, wd, dev(gl), epilogue=epilogue, clip=clip, h_save=h, ws=ws)
    assert M.read_status(ws) == 0
    return y, h


@pytest.mark.parametrize("M_,K,N,E,n_empty,seed", [
    (64, 128, 256, 4, 1, 0),       # one tile, one empty group
    (300, 192, 320, 5, 2, 1),      # partial row tiles, N not a multiple of 256, K = 3 blocks
    (1000, 256, 512, 9, 3, 2),     # many short groups
    (2500, 512, 768, 3, 0, 3),     # long groups, 3 column tiles
    (129, 64, 64, 1, 0, 4),        # single expert, one row past a tile
])
def test_forward_ragged(M_, K, N, E, n_empty, seed):
    rng = np.random.default_rng(seed)
    gl = counts_with_empties(rng, E, M_, n_empty)
    x = normal_bf16(rng, (M_, K))
    w = normal_bf16(rng, (E, K, N), 1 / np.sqrt(K))
    y, _ = gpu_forward(x, w, gl)
    assert_close("y", y, O.gmm_forward(f64(x), f64(w), gl))


# Shapes whose groups average >= 512 rows take the CTA-pair kernel (256-row
# tiles) for forward and dX; these cases put a 1-row group, a group shorter than
# one CTA's 128 rows, empty groups and partial column tiles on that path.
PAIR_CASES = [
    ([1700, 1, 130, 300], 192, 320),
    ([2048, 0, 0, 1], 256, 512),
    ([700, 900, 0, 600, 520], 128, 768),
    ([4096], 1024, 256),
]


@pytest.mark.parametrize("counts,K,N", PAIR_CASES)
def test_forward_and_dx_pair_path(counts, K, N):
    rng = np.random.default_rng(sum(counts) + K)
    gl = np.array(counts, np.int64)
    M_ = int(gl.sum())
    assert M_ >= 512 * len(gl)
    x = normal_bf16(rng, (M_, K))
    w = normal_bf16(rng, (len(gl), K, N), 1 / np.sqrt(K))
    dy = normal_bf16(rng, (M_, N))
    y, _ = gpu_forward(x, w, gl)
    assert_close("y", y, O.gmm_forward(f64(x), f64(w), gl))
    dx, dw = gpu_backward(x, w, gl, dy)
    dx_o, dw_o = O.gmm_backward(f64(x), f64(w), gl, f64(dy))
    assert_close("dx", dx, dx_o)
    assert_close("dw", dw, dw_o)


# Weight gradients whose groups have unequal depths, small enough for the
# CTA-pair kernel to give each group its own run of clusters (with dX's tiles
# as one more run when dX and dW share a launch), and a single group of deep
# tiles; one workspace serves every call, a permute included.
BALANCE_CASES = [
    ([512], 4096, 256),
    ([3803, 2000, 1000, 0], 1024, 2048),
    ([551, 443, 1656, 1018, 721, 0, 0, 3803], 1024, 2048),
    # dX and dW in one launch without the by-group schedule: more than 31 groups
    # with rows, and operands past the L2 budget; the clusters split between the two
    ([0, 0] + [520 + 7 * i for i in range(38)], 256, 256),
    ([30000, 20000, 15000, 5000], 256, 256),
]


@pytest.mark.parametrize("counts,K,N", BALANCE_CASES)
def test_weight_gradient_schedules(counts, K, N):
    import torch
    import moe_routed_expert_gb300 as M
    rng = np.random.default_rng(sum(counts) + 7 * K)
    gl = np.array(counts, np.int64)
    M_ = int(gl.sum())
    x = normal_bf16(rng, (M_, K))
    w = normal_bf16(rng, (len(gl), K, N), 1 / np.sqrt(K))
    dy = normal_bf16(rng, (M_, N))
    xd, wd, gld, dyd = dev_bf16(x), dev_bf16(w), dev(gl), dev_bf16(dy)
    ws = M.Workspace(max(M.gmm_workspace_size(M_, K, N, len(gl)), M.moe_permute_workspace_size(4096, 8, 64)))
    ids = torch.from_numpy(rng.integers(0, 64, size=(4096, 8)).astype(np.int32)).cuda()
    outs = []
    for _ in range(2):
        M.moe_permute(None, ids, 64, ws=ws)
        y = M.gmm_forward(xd, wd, gld, ws=ws)
        dx, dw = M.gmm_backward(xd, wd, gld, dyd, ws=ws)
        outs.append((y, dx, dw))
    assert M.read_status(ws) == 0
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    y, dx, dw = outs[0]
    assert_close("y", y, O.gmm_forward(f64(x), f64(w), gl))
    dx_o, dw_o = O.gmm_backward(f64(x), f64(w), gl, f64(dy))
    assert_close("dx", dx, dx_o)
    assert_close("dw", dw, dw_o)


def test_backward_results_feed_the_next_launch():
    """dX and dW of a small gmm_backward run side by side; the launch right
    behind it on the stream (a forward over dX, then over dW's first expert)
    must see both finished."""
    import torch
    import moe_routed_expert_gb300 as M
    rng = np.random.default_rng(41)
    gl = np.array([700, 0, 1300, 520, 1550], np.int64)
    K, N = 512, 1024
    M_ = int(gl.sum())
    x = normal_bf16(rng, (M_, K))
    w = normal_bf16(rng, (len(gl), K, N), 1 / np.sqrt(K))
    dy = normal_bf16(rng, (M_, N))
    w2 = normal_bf16(rng, (len(gl), K, 256), 1 / np.sqrt(K))
    w3 = normal_bf16(rng, (1, K, 64), 1 / np.sqrt(K))
    one = np.array([N], np.int64)
    dx_o, dw_o = O.gmm_backward(f64(x), f64(w), gl, f64(dy))
    ws = M.Workspace(256)
    for _ in range(3):
        dx, dw = M.gmm_backward(dev_bf16(x), dev_bf16(w), dev(gl), dev_bf16(dy), ws=ws)
        y2 = M.gmm_forward(dx, dev_bf16(w2), dev(gl), ws=ws)                        # reads dX at once
        y3 = M.gmm_forward(dw[0].t().contiguous(), dev_bf16(w3), dev(one), ws=ws)   # reads dW
        assert M.read_status(ws) == 0
        assert_close("dx", dx, dx_o)
        assert_close("dw", dw, dw_o)
        assert_close("forward over dx", y2, O.gmm_forward(host_f64(dx), f64(w2), gl))
        assert_close("forward over dw[0]^T", y3, O.gmm_forward(host_f64(dw)[0].T.copy(), f64(w3), one))


@pytest.mark.parametrize("clip", [0.0, 2.0])
def test_swiglu_epilogue_pair_path(clip):
    rng = np.random.default_rng(17)
    gl = np.array([1500, 3, 0, 1100], np.int64)
    K, I = 256, 384
    M_ = int(gl.sum())
    x = normal_bf16(rng, (M_, K))
    w = normal_bf16(rng, (len(gl), K, 2 * I), 2 / np.sqrt(K))
    a, h = gpu_forward(x, w, gl, epilogue=1, clip=clip, want_h=True)
    h_o = O.gmm_forward(f64(x), f64(w), gl)
    assert_close("h", h, h_o)
    assert_close("a(own h)", a, O.swiglu(host_f64(h), clip))
    # without h_save the activation is the same, bit for bit
    a2, _ = gpu_forward(x, w, gl, epilogue=1, clip=clip, want_h=False)
    assert np.array_equal(host_f64(a2), host_f64(a))


@pytest.mark.parametrize("M_,gl", [(200, [50, 0, 90]), (4000, [1500, 0, 600])])   # 128-row and pair kernels
def test_forward_rows_past_the_group_sum_are_untouched(M_, gl):
    import torch
    import moe_routed_expert_gb300 as M
    rng = np.random.default_rng(9)
    E, K, N = 3, 128, 256
    gl = np.array(gl, np.int64)     # sum below the rows in the buffer
    x = normal_bf16(rng, (M_, K))
    w = normal_bf16(rng, (E, K, N), 1 / np.sqrt(K))
    y = torch.full((M_, N), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = M.Workspace(256)
    M.gmm_forward(dev_bf16(x), dev_bf16(w), dev(gl), y=y, ws=ws)
    assert M.read_status(ws) == 0
    S = int(gl.sum())
    assert_close("y", y[:S], O.gmm_forward(f64(x[:S]), f64(w), gl))
    assert torch.all(y[S:] == 7.0)


@pytest.mark.parametrize("clip", [0.0, 1.5])
def test_forward_swiglu_epilogue(clip):
    rng = np.random.default_rng(11)
    E, K, I, M_ = 6, 256, 384, 777
    gl = counts_with_empties(rng, E, M_, 2)
    x = normal_bf16(rng, (M_, K))
    w = normal_bf16(rng, (E, K, 2 * I), 2 / np.sqrt(K))
    a, h = gpu_forward(x, w, gl, epilogue=1, clip=clip, want_h=True)
    h_o = O.gmm_forward(f64(x), f64(w), gl)
    assert_close("h", h, h_o)
    # the activation is taken on the stored bf16 H: compare on the GPU's own H too
    assert_close("a(own h)", a, O.swiglu(host_f64(h), clip))
    assert_close("a", a, O.swiglu(h_o, clip))


def test_workload_gmm_tiny_e4():
    wl = WORKLOADS["gmm_tiny_e4"]
    inp = gmm_inputs(wl)
    assert inp["group_list"][2] == 0 and inp["group_list"].sum() == wl.M
    y, _ = gpu_forward(inp["x"], inp["w"], inp["group_list"])
    assert_close("y", y, O.gmm_forward(f64(inp["x"]), f64(inp["w"]), inp["group_list"]))


def gpu_backward(x, w, gl, dy):
    import moe_routed_expert_gb300 as M
    ws = M.Workspace(256)
    dx, dw = M.gmm_backward(dev_bf16(x), dev_bf16(w), dev(gl), dev_bf16(dy), ws=ws)
    assert M.read_status(ws) == 0
    return dx, dw


@pytest.mark.parametrize("M_,K,N,E,n_empty,seed", [
    (64, 128, 256, 4, 1, 20),
    (300, 192, 320, 5, 2, 21),     # dW row tile past K, columns past N, partial 64-row blocks
    (1000, 256, 512, 9, 3, 22),
    (2500, 512, 768, 3, 0, 23),
])
def test_backward_ragged(M_, K, N, E, n_empty, seed):
    rng = np.random.default_rng(seed)
    gl = counts_with_empties(rng, E, M_, n_empty)
    x = normal_bf16(rng, (M_, K))
    w = normal_bf16(rng, (E, K, N), 1 / np.sqrt(K))
    dy = normal_bf16(rng, (M_, N))
    dx, dw = gpu_backward(x, w, gl, dy)
    dx_o, dw_o = O.gmm_backward(f64(x), f64(w), gl, f64(dy))
    assert_close("dx", dx, dx_o)
    assert_close("dw", dw, dw_o)
    for e in np.flatnonzero(gl == 0):
        assert np.all(host_f64(dw[e]) == 0)


def test_max_experts_forward_and_backward():
    """1024 experts, the most the library takes (its per-expert shared-memory
    tables are then full): a decode-like spread of 0-4 rows each, most empty,
    one group of 300 rows, and the last expert holding the final rows."""
    rng = np.random.default_rng(31)
    E, K, N = 1024, 128, 256
    gl = rng.choice([0, 0, 0, 1, 2, 4], size=E).astype(np.int64)
    gl[517] = 300
    gl[E - 1] = 3
    M_ = int(gl.sum())
    x = normal_bf16(rng, (M_, K))
    w = normal_bf16(rng, (E, K, N), 1 / np.sqrt(K))
    dy = normal_bf16(rng, (M_, N))
    y, _ = gpu_forward(x, w, gl)
    assert_close("y", y, O.gmm_forward(f64(x), f64(w), gl))
    dx, dw = gpu_backward(x, w, gl, dy)
    dx_o, dw_o = O.gmm_backward(f64(x), f64(w), gl, f64(dy))
    assert_close("dx", dx, dx_o)
    assert_close("dw", dw, dw_o)
    assert np.all(host_f64(dw)[gl == 0] == 0)


def test_workload_gmm_zipf_e8():
    wl = WORKLOADS["gmm_zipf_e8"]
    inp = gmm_inputs(wl)
    gl = inp["group_list"]
    assert (gl == 0).sum() == 2 and gl.sum() == wl.M
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    y, _ = gpu_forward(x, w, gl)
    dx, dw = gpu_backward(x, w, gl, dy)
    assert_close("y", y, O.gmm_forward(f64(x), f64(w), gl))
    dx_o, dw_o = O.gmm_backward(f64(x), f64(w), gl, f64(dy))
    assert_close("dx", dx, dx_o)
    assert_close("dw", dw, dw_o)


@pytest.mark.parametrize("bad,M_", [("negative", 64), ("too_many_rows", 64), ("negative", 4096),
                                     ("too_many_rows", 4096)])   # 128-row kernel, then CTA pairs
def test_bad_group_list_raises_device_status(bad, M_):
    import torch
    import moe_routed_expert_gb300 as M
    rng = np.random.default_rng(3)
    x = normal_bf16(rng, (M_, 128))
    w = normal_bf16(rng, (4, 128, 256))
    q = M_ // 4
    gl = np.array([2 * q, -1, q, q]) if bad == "negative" else np.array([2 * q, 2 * q, q, q])
    ws = M.Workspace(256)
    y = torch.zeros(M_, 256, dtype=torch.bfloat16, device="cuda")
    M.gmm_forward(dev_bf16(x), dev_bf16(w), dev(gl), y=y, ws=ws)
    assert M.read_status(ws) == 5
    assert torch.all(y == 0)   # nothing was computed
    ws.reset()
    assert M.read_status(ws) == 0


@pytest.mark.parametrize("counts,K,N,clip", [
    ([300, 0, 211, 90], 256, 512, 0.0),          # 128-row kernel
    ([1700, 1, 130, 300], 128, 320, 0.0),        # CTA pairs, partial column tiles
    ([2048, 0, 900, 1200], 384, 256, 1.0),       # CTA pairs, clip
])
def test_dx_swiglu_fused_equals_dx_then_swiglu_backward(counts, K, N, clip):
    """gmm_backward_dx_swiglu == gmm_backward's dx followed by moe_swiglu_backward,
    bit for bit, and both match the oracle's SwiGLU gradient on the same dA."""
    import moe_routed_expert_gb300 as M
    rng = np.random.default_rng(K + N + len(counts))
    gl = np.array(counts, np.int64)
    M_ = int(gl.sum())
    dy = normal_bf16(rng, (M_, N))
    w = normal_bf16(rng, (len(gl), K, N), 1 / np.sqrt(N))
    h = normal_bf16(rng, (M_, 2 * K), 1.5)
    ws = M.Workspace(256)
    dyd, wd, hd, gld = dev_bf16(dy), dev_bf16(w), dev_bf16(h), dev(gl)
    dh = M.gmm_backward_dx_swiglu(dyd, wd, gld, hd, clip, ws=ws)
    da, _ = M.gmm_backward(dev_bf16(np.zeros((M_, K), np.uint16)), wd, gld, dyd, need_dw=False, ws=ws)
    dh_ref = M.moe_swiglu_backward(hd, da, clip, ws=ws)
    assert M.read_status(ws) == 0
    assert np.array_equal(host_f64(dh), host_f64(dh_ref))
    assert_close("dh", dh, O.swiglu_backward(f64(h), host_f64(da), clip))
    da_o, _ = O.gmm_backward(np.zeros((M_, K)), f64(w), gl, f64(dy))
    assert_close("da", da, da_o)


# ---------------------------------------------------------------- gated activation variants ([MegaMoE])
ACT_CASES = [("swiglu", [1.5]), ("swiglustep", [1.5]), ("swigluoai", []), ("swigluoai", [2.0, 1.2, 0.5]),
             ("situglu", [1.5]), ("situglu", [2.0, 0.8])]


@pytest.mark.parametrize("kind,params", ACT_CASES)
@pytest.mark.parametrize("counts", [[1500, 3, 0, 1100], [300, 90, 0, 150]])   # CTA pairs; 128-row kernel
def test_activation_epilogue(kind, params, counts):
    """The gate_up forward with each activation: H matches the oracle's product,
    A the oracle's activation of the stored H."""
    import moe_routed_expert_gb300 as M
    rng = np.random.default_rng(31 + sum(counts))
    gl = np.array(counts, np.int64)
    K, I = 256, 384
    M_ = int(gl.sum())
    x = normal_bf16(rng, (M_, K))
    w = normal_bf16(rng, (len(gl), K, 2 * I), 2 / np.sqrt(K))
    import torch
    h = torch.empty(M_, 2 * I, dtype=torch.bfloat16, device="cuda")
    ws = M.Workspace(256)
    a = M.gmm_forward(dev_bf16(x), dev_bf16(w), dev(gl), h_save=h, activation=(kind, params), ws=ws)
    assert M.read_status(ws) == 0
    assert_close("h", h, O.gmm_forward(f64(x), f64(w), gl))
    assert_close("a", a, O.gated_activation(host_f64(h), O.activation(kind, params)))
    # without h_save the activation is the same, bit for bit
    a2 = M.gmm_forward(dev_bf16(x), dev_bf16(w), dev(gl), activation=(kind, params), ws=ws)
    assert np.array_equal(host_f64(a2), host_f64(a))


@pytest.mark.parametrize("kind,params", ACT_CASES)
@pytest.mark.parametrize("counts,K,N", [([300, 0, 211, 90], 256, 512), ([2048, 0, 900, 1200], 384, 256)])
def test_activation_gradient_fused_in_dx(kind, params, counts, K, N):
    """The dX epilogue's activation gradient == dx then moe_activation_backward,
    bit for bit, and both match the oracle's gradient on the same dA."""
    import moe_routed_expert_gb300 as M
    rng = np.random.default_rng(K + N + len(counts) + len(kind))
    gl = np.array(counts, np.int64)
    M_ = int(gl.sum())
    dy = normal_bf16(rng, (M_, N))
    w = normal_bf16(rng, (len(gl), K, N), 1 / np.sqrt(N))
    h = normal_bf16(rng, (M_, 2 * K), 1.5)
    ws = M.Workspace(256)
    dyd, wd, hd, gld = dev_bf16(dy), dev_bf16(w), dev_bf16(h), dev(gl)
    dh = M.gmm_backward_dx_swiglu(dyd, wd, gld, hd, activation=(kind, params), ws=ws)
    da, _ = M.gmm_backward(dev_bf16(np.zeros((M_, K), np.uint16)), wd, gld, dyd, need_dw=False, ws=ws)
    dh_ref = M.moe_swiglu_backward(hd, da, activation=(kind, params), ws=ws)
    assert M.read_status(ws) == 0
    assert np.array_equal(host_f64(dh), host_f64(dh_ref))
    assert_close("dh", dh, O.gated_activation_backward(f64(h), host_f64(da), O.activation(kind, params)))


# ---------------------------------------------------------------- transposed weights ([MegaMoE] transposeWeight)
@pytest.mark.parametrize("counts,K,N", [([300, 0, 211, 90], 256, 512),      # 128-row kernel
                                        ([2048, 0, 900, 1200], 384, 512)])  # CTA pairs
def test_transposed_weights(counts, K, N):
    """w stored [E, N, K]: forward (plain and SwiGLU), dX (plain and with the
    activation gradient) and dW (written [E, N, K]) against the oracle on W."""
    import torch
    import moe_routed_expert_gb300 as M
    rng = np.random.default_rng(K + N + 5)
    gl = np.array(counts, np.int64)
    M_ = int(gl.sum())
    x = normal_bf16(rng, (M_, K))
    w = normal_bf16(rng, (len(gl), K, N), 1 / np.sqrt(K))
    dy = normal_bf16(rng, (M_, N))
    wt = np.ascontiguousarray(np.transpose(w, (0, 2, 1)))      # [E, N, K]
    xd, wtd, gld, dyd = dev_bf16(x), dev_bf16(wt), dev(gl), dev_bf16(dy)
    ws = M.Workspace(256)
    y = M.gmm_forward(xd, wtd, gld, w_transposed=True, ws=ws)
    assert_close("y", y, O.gmm_forward(f64(x), f64(w), gl))
    h = torch.empty(M_, N, dtype=torch.bfloat16, device="cuda")
    a = M.gmm_forward(xd, wtd, gld, activation=("swigluoai", []), h_save=h, w_transposed=True, ws=ws)
    assert_close("h", h, O.gmm_forward(f64(x), f64(w), gl))
    assert_close("a", a, O.gated_activation(host_f64(h), O.activation("swigluoai")))
    dx, dwt = M.gmm_backward(xd, wtd, gld, dyd, w_transposed=True, ws=ws)
    assert tuple(dwt.shape) == (len(gl), N, K)
    dx_o, dw_o = O.gmm_backward(f64(x), f64(w), gl, f64(dy))
    assert_close("dx", dx, dx_o)
    assert_close("dw^T", dwt, np.transpose(dw_o, (0, 2, 1)))
    # dX over the transposed down weights with the activation gradient: w2^T [E, N, I]
    I = K // 2
    w2 = normal_bf16(rng, (len(gl), I, N), 1 / np.sqrt(N))
    hh = normal_bf16(rng, (M_, 2 * I), 1.5)
    w2t = dev_bf16(np.ascontiguousarray(np.transpose(w2, (0, 2, 1))))
    dh = M.gmm_backward_dx_swiglu(dyd, w2t, gld, dev_bf16(hh), activation=("situglu", [1.5]), w_transposed=True,
                                  ws=ws)
    da, _ = M.gmm_backward(dev_bf16(np.zeros((M_, I), np.uint16)), w2t, gld, dyd, need_dw=False, w_transposed=True,
                           ws=ws)
    assert M.read_status(ws) == 0
    assert_close("da", da, O.gmm_backward(np.zeros((M_, I)), f64(w2), gl, f64(dy))[0])
    assert_close("dh", dh, O.gated_activation_backward(f64(hh), host_f64(da), O.activation("situglu", [1.5])))
