"""CUDA-graph capture of the layer forward (decode sizes).  Every entry point is
stream-ordered, with no host synchronisation and its TMA descriptors passed by
value as kernel parameters, so one call can be captured into a graph (the
programmatic-launch attribute becomes a programmatic graph edge) and replayed
on new inputs copied into the captured buffers.  Replays must equal eager calls
bit for bit, across different inputs and repeated replays."""
import numpy as np
import pytest

from tests._util import dev, dev_bf16
from workloads import WORKLOADS, layer_inputs, mx_layer_weights, pack_fp4

pytestmark = pytest.mark.gpu


def _inputs(wl, seed):
    return layer_inputs(wl, seed=seed, with_weights=False)


@pytest.mark.parametrize("name", ["layer_decode_t64", "layer_decode_mx_t64", "layer_decode_a8w4_t64",
                                  "layer_decode_a4w4_t64"])
def test_layer_forward_replays_from_a_cuda_graph(name):
    import torch
    import moe_routed_expert_gb300 as M
    wl = WORKLOADS[name]
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    if wl.mx:
        wts = mx_layer_weights(wl)
        wf = wl.w_mx or wl.mx
        pk = pack_fp4 if wf == "e2m1" else (lambda a: a)
        w1q, w2q = dev(pk(wts["w1_q"])), dev(pk(wts["w2_q"]))
        w1s, w2s = dev(wts["w1_s"]), dev(wts["w2_s"])
        ws = M.Workspace(M.moe_layer_mx_workspace_size(T, H, I, E, k))

        def layer(x, ids, tw, y):
            M.moe_layer_forward_mx(x, ids, tw, w1q, w1s, w2q, w2s, x_fmt=wl.mx, w_fmt=wf, y=y, ws=ws)
    else:
        full = layer_inputs(wl)
        w1, w2 = dev_bf16(full["w1"]), dev_bf16(full["w2"])
        ws = M.Workspace(M.moe_layer_workspace_size(T, H, I, E, k))

        def layer(x, ids, tw, y):
            M.moe_layer_forward(x, ids, tw, w1, w2, wl.clip, y=y, ws=ws)

    # static buffers the graph reads and writes
    first = _inputs(wl, 101)
    x = dev_bf16(first["x"])
    ids = dev(first["topk_ids"])
    tw = dev(first["topk_w"])
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    layer(x, ids, tw, y)               # eager warm-up: first-call set-up happens outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            layer(x, ids, tw, y)
    torch.cuda.current_stream().wait_stream(s)
    for seed in (101, 202, 303):
        inp = _inputs(wl, seed)
        x.copy_(dev_bf16(inp["x"]))
        ids.copy_(dev(inp["topk_ids"]))
        tw.copy_(dev(inp["topk_w"]))
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        y_graph = y.clone()
        y_eager = torch.empty_like(y)
        layer(x, ids, tw, y_eager)
        torch.cuda.synchronize()
        assert M.read_status(ws) == 0
        assert torch.equal(y_graph, y_eager), seed
        assert torch.isfinite(y_graph.float()).all()
