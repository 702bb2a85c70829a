"""The fused layer forward ("MegaMoE", 算子功能: dispatch, the expert matmuls
and the combine as one operator) against the unfused chain and the oracle.

* gmm_forward_gather_act (rows fetched from x through the permutation) must
  equal gmm_forward with the activation on the permuted rows, bit for bit:
  the same products in the same order, only the rows' source differs.
* gmm_forward_combine must equal gmm_forward followed by moe_unpermute, bit
  for bit: the same slot order and the same fp32 arithmetic.
* moe_layer_forward without saved tensors (the fused path) must equal the
  layer with saved tensors (the unfused path) bit for bit, and y must match
  the oracle end to end (a token's output sums its k slots; see the layer
  tests for the step-by-step checks of the same kernels).
Cases cover empty experts, unused (-1) slots, tokens with no routed slot,
slot counts above eight, widths that end inside a 256-column tile, the
transposed weight layouts and the pages' other activations."""
import numpy as np
import pytest

import oracle as O
from tests._util import assert_close, dev, dev_bf16, f64, host_f64
from workloads import WORKLOADS, LayerWorkload, layer_inputs

pytestmark = pytest.mark.gpu


def _inputs(wl, unused=0.0, dead_tokens=(), drop_expert=None, seed=7):
    inp = layer_inputs(wl)
    ids = inp["topk_ids"]
    rng = np.random.default_rng(seed)
    if unused:
        ids[rng.random(ids.shape) < unused] = -1
    if drop_expert is not None:
        ids[ids == drop_expert] = -1
    for t in dead_tokens:
        ids[t, :] = -1
    return inp


CASES = [
    # name, T, H, E, k, I, unused-slot fraction, tokens with no slot, expert nobody picks
    ("tiny_e4", 48, 128, 4, 2, 128, 0.0, (), None),
    ("ragged", 333, 384, 16, 4, 256, 0.15, (0, 5, 332), 3),
    ("k6_h320", 257, 320, 12, 6, 128, 0.1, (7,), None),
    ("k10", 130, 256, 24, 10, 128, 0.05, (), 0),
    ("e64_sparse", 64, 512, 64, 8, 128, 0.0, (), None),
]


def _wl(c):
    name, T, H, E, k, I = c[:6]
    return LayerWorkload(name, 40 + len(name), T=T, H=H, E=E, k=k, I=I, clip=0.0, hot_bias=0.0, backward=False)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("w_transposed", [False, True], ids=["w", "wT"])
def test_gather_act_and_combine_equal_the_unfused_ops(case, w_transposed):
    import torch
    import moe_routed_expert_gb300 as M
    wl = _wl(case)
    inp = _inputs(wl, *case[6:])
    x, ids, tw = dev_bf16(inp["x"]), dev(inp["topk_ids"]), dev(inp["topk_w"])
    w1, w2 = dev_bf16(inp["w1"]), dev_bf16(inp["w2"])
    if w_transposed:
        w1, w2 = w1.transpose(1, 2).contiguous(), w2.transpose(1, 2).contiguous()
    x_perm, gl, rmap, sflat = M.moe_permute(x, ids, wl.E)
    R = int(gl.sum())
    act = ("swiglu", [0.0])
    # gate_up: gathered rows vs the permuted rows
    a_ref = M.gmm_forward(x_perm, w1, gl, activation=act, w_transposed=w_transposed)
    a_got = torch.full_like(a_ref, 7.0)
    M.gmm_forward_gather_act(x, sflat, wl.k, w1, gl, act, y=a_got, w_transposed=w_transposed)
    torch.cuda.synchronize()
    assert torch.equal(a_got[:R], a_ref[:R])
    assert torch.all(a_got[R:] == 7.0)          # rows past the groups are not written
    # down + combine vs down then the standalone combine
    y2 = M.gmm_forward(a_ref, w2, gl, w_transposed=w_transposed)
    y_ref = M.moe_unpermute(y2, rmap, tw, wl.T, wl.k)
    y_got = torch.full_like(y_ref, 5.0)
    ws = M.Workspace(M.gmm_forward_combine_workspace_size(wl.T, wl.k, wl.T * wl.k, wl.H))
    for _ in range(2):   # twice: the arrival counts start at zero on every call
        M.gmm_forward_combine(a_ref, w2, gl, rmap, sflat, tw, y=y_got, w_transposed=w_transposed, ws=ws)
        assert M.read_status(ws) == 0
        assert torch.equal(y_got, y_ref)
    for t in case[7]:
        assert torch.all(y_got[t] == 0)


def _layer(inp, wl, saved, act=None, w_flags=0, w1=None, w2=None):
    import moe_routed_expert_gb300 as M
    x, ids, tw = dev_bf16(inp["x"]), dev(inp["topk_ids"]), dev(inp["topk_w"])
    w1 = dev_bf16(inp["w1"]) if w1 is None else w1
    w2 = dev_bf16(inp["w2"]) if w2 is None else w2
    ws = M.Workspace(M.moe_layer_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.k))
    sv = M.LayerSaved(wl.T, wl.H, wl.I, wl.E, wl.k) if saved else None
    y = M.moe_layer_forward(x, ids, tw, w1, w2, wl.clip, saved=sv, activation=act, w_flags=w_flags, ws=ws)
    assert M.read_status(ws) == 0
    return y


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fused_layer_forward_small(case):
    import torch
    wl = _wl(case)
    inp = _inputs(wl, *case[6:])
    y_fused = _layer(inp, wl, saved=False)
    y_unfused = _layer(inp, wl, saved=True)
    assert torch.equal(y_fused, y_unfused)
    assert torch.equal(_layer(inp, wl, saved=False), y_fused)      # deterministic
    y_o, _ = O.moe_layer_forward(f64(inp["x"]), inp["topk_ids"], inp["topk_w"], f64(inp["w1"]), f64(inp["w2"]),
                                 wl.clip)
    assert_close("y (fused, end to end)", y_fused, y_o)


@pytest.mark.parametrize("act", [("swiglu", [7.0]), ("swiglustep", [0.8]), ("swigluoai", [7.0, 1.702, 1.0]),
                                 ("situglu", [1.0, 2.0])], ids=lambda a: a[0])
def test_fused_layer_forward_activations_and_layouts(act):
    import torch
    wl = _wl(CASES[1])
    inp = _inputs(wl, *CASES[1][6:])
    y_fused = _layer(inp, wl, saved=False, act=act)
    assert torch.equal(y_fused, _layer(inp, wl, saved=True, act=act))
    w1t = dev_bf16(np.ascontiguousarray(np.transpose(inp["w1"], (0, 2, 1))))
    w2t = dev_bf16(np.ascontiguousarray(np.transpose(inp["w2"], (0, 2, 1))))
    assert torch.equal(_layer(inp, wl, saved=False, act=act, w_flags=3, w1=w1t, w2=w2t), y_fused)
    y_o, _ = O.moe_layer_forward(f64(inp["x"]), inp["topk_ids"], inp["topk_w"], f64(inp["w1"]), f64(inp["w2"]),
                                 wl.clip, act=O.activation(*act))
    assert_close("y (fused, end to end)", y_fused, y_o)


@pytest.mark.parametrize("name", ["layer_decode_t64", "layer_prefill_t4096"])
def test_fused_layer_forward_workloads(name):
    """The prefill and decode layer workloads, every output: the fused forward
    equals the unfused one bit for bit and the oracle end to end."""
    import torch
    wl = WORKLOADS[name]
    inp = layer_inputs(wl)
    y_fused = _layer(inp, wl, saved=False)
    assert torch.equal(y_fused, _layer(inp, wl, saved=True))
    y_o, _ = O.moe_layer_forward(f64(inp["x"]), inp["topk_ids"], inp["topk_w"], f64(inp["w1"]), f64(inp["w2"]),
                                 wl.clip)
    assert_close("y (fused, end to end)", y_fused, y_o)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_expert_mlp_one_launch_equals_the_two_gmms(case):
    """moe_expert_mlp_forward (both expert matmuls in one launch, gate_up rows
    gathered from x) against gmm_forward with the activation on the permuted
    rows and gmm_forward: bit for bit, rows past the groups untouched, and the
    same on a second call (its readiness counts start at zero each time)."""
    import torch
    import moe_routed_expert_gb300 as M
    wl = _wl(case)
    inp = _inputs(wl, *case[6:])
    x, ids = dev_bf16(inp["x"]), dev(inp["topk_ids"])
    w1, w2 = dev_bf16(inp["w1"]), dev_bf16(inp["w2"])
    x_perm, gl, rmap, sflat = M.moe_permute(x, ids, wl.E)
    R = int(gl.sum())
    act = ("swiglu", [3.0])
    a_ref = M.gmm_forward(x_perm, w1, gl, activation=act)
    y2_ref = M.gmm_forward(a_ref, w2, gl)
    a = torch.full_like(a_ref, 7.0)
    y2 = torch.full_like(y2_ref, 5.0)
    ws = M.Workspace(M.moe_expert_mlp_workspace_size(wl.T, wl.k, wl.E))
    for _ in range(2):
        M.moe_expert_mlp_forward(x, sflat, gl, w1, w2, wl.k, act, a=a, y2=y2, ws=ws)
        assert M.read_status(ws) == 0
        assert torch.equal(a[:R], a_ref[:R]) and torch.equal(y2[:R], y2_ref[:R])
        assert torch.all(a[R:] == 7.0) and torch.all(y2[R:] == 5.0)


def test_expert_mlp_one_launch_at_the_prefill_size():
    import torch
    import moe_routed_expert_gb300 as M
    wl = WORKLOADS["layer_prefill_t4096"]
    inp = layer_inputs(wl)
    x, ids = dev_bf16(inp["x"]), dev(inp["topk_ids"])
    w1, w2 = dev_bf16(inp["w1"]), dev_bf16(inp["w2"])
    x_perm, gl, rmap, sflat = M.moe_permute(x, ids, wl.E)
    a_ref = M.gmm_forward(x_perm, w1, gl, epilogue=1)
    y2_ref = M.gmm_forward(a_ref, w2, gl)
    a, y2 = M.moe_expert_mlp_forward(x, sflat, gl, w1, w2, wl.k)
    torch.cuda.synchronize()
    assert torch.equal(a, a_ref) and torch.equal(y2, y2_ref)
