"""Parity of the combine-side kernels (weighted combine, its token and probs
gradients, the permute's token gradient, the SwiGLU gradient) with the
oracle, within the pages' bf16 tolerance; unused (-1) slots included."""
import numpy as np
import pytest

import oracle as O
from tests._util import assert_close, dev, dev_bf16, f64, host_f64
from workloads import normal_bf16

pytestmark = pytest.mark.gpu


def routed(rng, T, k, E, p_unused):
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[rng.random(ids.shape) < p_unused] = -1
    w = rng.random((T, k)).astype(np.float32)
    rmap, sflat, counts, _ = O.stable_counting_sort(ids, E)
    return ids, w, rmap, int(counts.sum())


@pytest.mark.parametrize("T,k,E,H,p", [(1, 1, 1, 64, 0.0), (37, 3, 8, 200, 0.3), (500, 8, 64, 2048, 0.1),
                                       (300, 8, 16, 4096, 0.0), (64, 16, 32, 2120, 0.25)])
def test_unpermute_and_gradients(T, k, E, H, p):
    import moe_routed_expert_gb300 as M
    rng = np.random.default_rng(T + H)
    ids, w, rmap, R = routed(rng, T, k, E, p)
    yp = normal_bf16(rng, (T * k, H))      # rows past R are never read
    dy = normal_bf16(rng, (T, H))
    ws = M.Workspace(256)
    y = M.moe_unpermute(dev_bf16(yp), dev(rmap), dev(w), T, k, ws=ws)
    dyp, dpr = M.moe_unpermute_backward(dev_bf16(dy), dev_bf16(yp), dev(rmap), dev(w), k, ws=ws)
    dx = M.moe_permute_backward(dev_bf16(yp), dev(rmap), T, k, ws=ws)
    assert M.read_status(ws) == 0
    assert_close("y", y, O.moe_unpermute(f64(yp[:R]), rmap, w, T, k))
    dyp_o, dpr_o = O.moe_unpermute_backward(f64(dy), f64(yp[:R]), rmap, w, T, k)
    assert_close("dy_perm", host_f64(dyp)[:R], dyp_o)
    assert_close("dprobs", dpr, dpr_o)
    assert_close("dx", dx, O.moe_permute_backward(f64(yp[:R]), rmap, T, k))


def test_bad_row_ids_raise_device_status():
    import moe_routed_expert_gb300 as M
    rng = np.random.default_rng(1)
    T, k, H = 4, 2, 64
    yp = normal_bf16(rng, (T * k, H))
    rmap = np.array([0, 1, 2, 3, 4, 5, 6, 99], np.int32)
    ws = M.Workspace(256)
    M.moe_unpermute(dev_bf16(yp), dev(rmap), dev(np.ones((T, k), np.float32)), T, k, ws=ws)
    assert M.read_status(ws) == 5


@pytest.mark.parametrize("clip", [0.0, 7.0, 0.75])
def test_swiglu_backward(clip):
    import moe_routed_expert_gb300 as M
    rng = np.random.default_rng(int(clip * 100))
    rows, I = 1000, 384
    h = normal_bf16(rng, (rows, 2 * I), 2.0)
    da = normal_bf16(rng, (rows, I))
    ws = M.Workspace(256)
    dh = M.moe_swiglu_backward(dev_bf16(h), dev_bf16(da), clip, ws=ws)
    assert M.read_status(ws) == 0
    assert_close("dh", dh, O.swiglu_backward(f64(h), f64(da), clip))
