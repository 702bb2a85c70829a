"""Parity of the CUDA permute (histogram, scan, stable counting-sort scatter,
row gather) with the oracle: bit-exact for every integer output and for the
permuted rows (a copy).  Cases up to 1024 slots take the one-block index
kernel, larger ones the three-kernel path (count, rank, gather)."""
import json
import os

import numpy as np
import pytest

import oracle as O
from tests._util import dev, dev_bf16, host_f64
from workloads import WORKLOADS, layer_inputs, normal_bf16

pytestmark = pytest.mark.gpu


def run_permute(x_bits, ids, E):
    import moe_routed_expert_gb300 as M
    ws = M.Workspace(M.moe_permute_workspace_size(ids.shape[0], ids.shape[1], E))
    out = M.moe_permute(dev_bf16(x_bits) if x_bits is not None else None, dev(ids), E, ws=ws)
    st = M.read_status(ws)
    return out, st


def check_against_oracle(x_bits, ids, E):
    (x_perm, gl, rmap, sflat), st = run_permute(x_bits, ids, E)
    assert st == 0
    r_o, s_o, c_o, _ = O.stable_counting_sort(ids, E)
    R = int(c_o.sum())
    np.testing.assert_array_equal(gl.cpu().numpy(), c_o)
    np.testing.assert_array_equal(rmap.cpu().numpy(), r_o)
    sf = sflat.cpu().numpy()
    np.testing.assert_array_equal(sf[:R], s_o)
    assert np.all(sf[R:] == -1)
    if x_bits is not None:
        k = ids.shape[1]
        got = x_perm[:R].cpu().view(dtype=__import__("torch").int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(got, x_bits[s_o.astype(np.int64) // k])
    return R


def test_worked_example():
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "gmm_worked_example.json")))
    ids = np.array([[1, 3], [1, -1], [0, -1], [3, -1]], np.int32)
    x = normal_bf16(np.random.default_rng(0), (4, 64))
    (xp, gl, rmap, sflat), st = run_permute(x, ids, 4)
    assert st == 0
    assert gl.cpu().tolist() == g["group_list"]
    assert rmap.cpu().tolist() == [1, 3, 2, -1, 0, -1, 4, -1]
    assert sflat.cpu().tolist() == [4, 0, 2, 1, 6, -1, -1, -1]
    check_against_oracle(x, ids, 4)


@pytest.mark.parametrize("T,k,E,H,p_unused", [
    (1, 1, 1, 64, 0.0), (7, 3, 5, 72, 0.3), (33, 2, 4, 128, 0.5), (1000, 8, 256, 2048, 0.05),
    (3000, 4, 1024, 64, 0.1), (5000, 8, 64, 136, 0.0), (2049, 1, 3, 8, 0.0), (129, 64, 64, 64, 0.2),
    # either side of the one-block index path (up to 1024 slots), with 1024 experts
    (128, 8, 1024, 64, 0.1), (1025, 1, 7, 16, 0.2), (100, 8, 1024, 32, 0.0),
    # the prefill batch size (32768 slots) and around it: full, ragged, 1024 experts
    (4096, 8, 256, 32, 0.0), (32769, 1, 5, 16, 0.1), (4000, 8, 1024, 32, 0.3), (1057, 31, 40, 8, 0.05),
])
def test_random_ragged(T, k, E, H, p_unused):
    rng = np.random.default_rng(T * 7 + k)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) if k <= E else None
    ids[rng.random(ids.shape) < p_unused] = -1
    x = normal_bf16(rng, (T, H))
    check_against_oracle(x, ids, E)


def test_index_only_and_skewed():
    rng = np.random.default_rng(5)
    T, k, E = 4000, 8, 64
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    ids[:, 0] = 17  # one expert takes every token once
    check_against_oracle(None, ids, E)


@pytest.mark.parametrize("name", ["layer_prefill_t4096", "layer_decode_t64", "layer_train_t16384"])
def test_workload_routing_exact(name):
    wl = WORKLOADS[name]
    inp = layer_inputs(wl, with_weights=False)
    R = check_against_oracle(inp["x"], inp["topk_ids"], wl.E)
    assert R == wl.T * wl.k


def test_bad_ids_raise_device_status():
    ids = np.array([[0, 1], [2, 9]], np.int32)
    (_, _, rmap, _), st = run_permute(None, ids, 4)
    assert st == 5  # MOE_ERR_DEVICE
    assert rmap.cpu().tolist()[3] == -1
    ids = np.array([[0, -2]], np.int32)
    _, st = run_permute(None, ids, 4)
    assert st == 5


@pytest.mark.parametrize("T,k", [(2000, 4), (10000, 4)])
def test_bad_ids_raise_device_status_larger_batches(T, k):
    """The multi-block index path flags a bad id too, and treats it as an
    unused slot."""
    rng = np.random.default_rng(T)
    E = 16
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    ids[T // 2, 1] = E
    (_, _, rmap, _), st = run_permute(None, ids, E)
    assert st == 5  # MOE_ERR_DEVICE
    assert rmap.cpu().numpy()[(T // 2) * k + 1] == -1


def test_empty_tokens():
    import torch
    import moe_routed_expert_gb300 as M
    ids = torch.empty(0, 4, dtype=torch.int32, device="cuda")
    ws = M.Workspace(M.moe_permute_workspace_size(0, 4, 8))
    gl = torch.full((8,), 7, dtype=torch.int64, device="cuda")
    out = (None, gl, torch.empty(0, dtype=torch.int32, device="cuda"), torch.empty(0, dtype=torch.int32, device="cuda"))
    M.moe_permute(None, ids, 8, out=out, ws=ws)
    assert gl.cpu().tolist() == [0] * 8
    assert M.read_status(ws) == 0
