"""Parity of the whole routed-expert layer (forward, and forward + backward)
through the C ABI with the oracle.

Small cases compare every output.  The full workload sizes compare what the
oracle can compute in seconds without changing the result:
* every integer output (group_list, row_id_map, sorted_flat), bit-exact;
* y, dx and dprobs of a sample of tokens -- a token's outputs depend only on
  its own row and the weights, so the oracle runs on that token subset;
* dW1 and dW2 of a sample of experts -- an expert's weight gradient depends
  only on its own rows, so the oracle runs on the sub-problem whose other
  slots are marked unused (-1).
"""
import numpy as np
import pytest

import oracle as O
from tests._util import assert_close, dev, dev_bf16, f64, host_f64
from workloads import WORKLOADS, LayerWorkload, layer_inputs

pytestmark = pytest.mark.gpu


def gpu_layer(inp, wl, backward, want_saved=False):
    import moe_routed_expert_gb300 as M
    x, w1, w2 = dev_bf16(inp["x"]), dev_bf16(inp["w1"]), dev_bf16(inp["w2"])
    ids, tw = dev(inp["topk_ids"]), dev(inp["topk_w"])
    ws = M.Workspace(M.moe_layer_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.k))
    saved = M.LayerSaved(wl.T, wl.H, wl.I, wl.E, wl.k) if (backward or want_saved) else None
    y = M.moe_layer_forward(x, ids, tw, w1, w2, wl.clip, saved=saved, ws=ws)
    out = {"y": y, "saved": saved}
    if backward:
        dx, dw1, dw2, dpr = M.moe_layer_backward(dev_bf16(inp["dy"]), tw, w1, w2, saved, wl.clip, ws=ws)
        out.update(dx=dx, dw1=dw1, dw2=dw2, dprobs=dpr)
    assert M.read_status(ws) == 0
    return out


def oracle_layer(inp, wl, backward, tokens=None, keep_expert=None, wf=None):
    ids = inp["topk_ids"]
    sel = slice(None) if tokens is None else tokens
    ids = ids[sel].copy()
    if keep_expert is not None:
        ids[ids != keep_expert] = -1
    x, tw = f64(inp["x"][sel]), inp["topk_w"][sel]
    w1, w2 = wf if wf is not None else (f64(inp["w1"]), f64(inp["w2"]))
    y, sv = O.moe_layer_forward(x, ids, tw, w1, w2, wl.clip)
    out = {"y": y, "saved": sv}
    if backward:
        dx, dw1, dw2, dpr = O.moe_layer_backward(f64(inp["dy"][sel]), sv, tw, w1, w2, wl.clip)
        out.update(dx=dx, dw1=dw1, dw2=dw2, dprobs=dpr)
    return out


SMALL = [
    LayerWorkload("small_a", 31, T=200, H=256, E=8, k=2, I=128, clip=0.0, hot_bias=0.0, backward=True),
    LayerWorkload("small_b", 32, T=333, H=384, E=16, k=4, I=256, clip=7.0, hot_bias=2.0, backward=True),
    LayerWorkload("small_c", 33, T=64, H=512, E=64, k=8, I=128, clip=0.5, hot_bias=0.0, backward=True),
]


@pytest.mark.parametrize("wl", SMALL, ids=[w.name for w in SMALL])
def test_layer_small_every_output(wl):
    inp = layer_inputs(wl)
    if wl.name == "small_b":    # unused slots and an expert nobody picks
        inp["topk_ids"][::5, -1] = -1
        inp["topk_ids"][inp["topk_ids"] == 3] = -1
    g = gpu_layer(inp, wl, backward=True)
    o = oracle_layer(inp, wl, backward=True)
    sv, so = g["saved"], o["saved"]
    R = int(so["group_list"].sum())
    np.testing.assert_array_equal(sv.group_list.cpu().numpy(), so["group_list"])
    np.testing.assert_array_equal(sv.row_id_map.cpu().numpy(), so["row_id_map"])
    assert_close("h", host_f64(sv.h)[:R], so["h"])
    assert_close("a", host_f64(sv.a)[:R], so["a"])
    assert_close("y2", host_f64(sv.y2)[:R], so["y2"])
    for key in ("y", "dx", "dw1", "dw2", "dprobs"):
        assert_close(key, g[key], o[key])


@pytest.mark.parametrize("name", ["layer_decode_t64", "layer_prefill_t4096"])
def test_layer_forward_workloads_every_output(name):
    wl = WORKLOADS[name]
    inp = layer_inputs(wl)
    g = gpu_layer(inp, wl, backward=False, want_saved=True)
    o = oracle_layer(inp, wl, backward=False)
    np.testing.assert_array_equal(g["saved"].group_list.cpu().numpy(), o["saved"]["group_list"])
    assert_close("y", g["y"], o["y"])


def test_layer_train_t16384_sampled():
    wl = WORKLOADS["layer_train_t16384"]
    inp = layer_inputs(wl)
    g = gpu_layer(inp, wl, backward=True)
    sv = g["saved"]
    # integer outputs: exact, whole problem
    rmap_o, sflat_o, counts_o, _ = O.stable_counting_sort(inp["topk_ids"], wl.E)
    np.testing.assert_array_equal(sv.group_list.cpu().numpy(), counts_o)
    np.testing.assert_array_equal(sv.row_id_map.cpu().numpy(), rmap_o)
    np.testing.assert_array_equal(sv.sorted_flat.cpu().numpy(), sflat_o)
    # sampled tokens
    rng = np.random.default_rng(123)
    toks = np.sort(rng.choice(wl.T, size=48, replace=False))
    toks = np.concatenate([[0, wl.T - 1], toks])
    wf = (f64(inp["w1"]), f64(inp["w2"]))
    o = oracle_layer(inp, wl, backward=True, tokens=toks, wf=wf)
    for key in ("y", "dx", "dprobs"):
        assert_close(key + "[tokens]", host_f64(g[key])[toks], o[key])
    # sampled experts: the hot one, and two others
    hot = inp["hot_expert"]
    others = [e for e in rng.permutation(wl.E) if e != hot][:2]
    dw1, dw2 = host_f64(g["dw1"]), host_f64(g["dw2"])
    for e in [hot] + others:
        oe = oracle_layer(inp, wl, backward=True, keep_expert=e, wf=wf)
        assert_close("dw1[%d]" % e, dw1[e], oe["dw1"][e])
        assert_close("dw2[%d]" % e, dw2[e], oe["dw2"][e])
