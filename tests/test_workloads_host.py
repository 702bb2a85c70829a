"""The synthetic inputs (workloads.py) against the recipes they are documented
with: the tiny GMM's counts, the Zipf counts as the largest-remainder rounding of
Zipf(s) shares, and the routing's structure (distinct top-k ids per token,
renormalised weights, the hot expert of the training workload)."""
import numpy as np

from workloads import WORKLOADS, gmm_inputs, layer_inputs


def _largest_remainder(shares, total):
    raw = np.asarray(shares, np.float64) / np.sum(shares) * total
    out = np.floor(raw).astype(np.int64)
    for i in np.argsort(-(raw - out), kind="stable")[: total - out.sum()]:
        out[i] += 1
    return out


def test_tiny_gmm_counts():
    wl = WORKLOADS["gmm_tiny_e4"]
    gl = gmm_inputs(wl)["group_list"]
    assert gl.dtype == np.int64 and gl.shape == (4,)
    assert gl.sum() == 64 and gl[2] == 0 and np.all(gl[[0, 1, 3]] > 0)


def test_zipf_counts_are_rounded_zipf_shares():
    wl = WORKLOADS["gmm_zipf_e8"]
    gl = gmm_inputs(wl)["group_list"]
    assert gl.sum() == wl.M == 8192 and (gl == 0).sum() == 2
    live = np.sort(gl[gl > 0])[::-1]
    want = _largest_remainder([r ** -1.2 for r in range(1, 7)], 8192)
    assert live.tolist() == want.tolist() == [3803, 1656, 1018, 721, 551, 443]


def _check_routing(inp, E, k):
    ids, w = inp["topk_ids"], inp["topk_w"]
    assert ids.dtype == np.int32 and w.dtype == np.float32 and ids.shape == w.shape
    assert np.all((ids >= 0) & (ids < E))
    assert all(len(set(row)) == k for row in ids.tolist())        # top-k picks distinct experts
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-6) and np.all(w > 0)
    assert np.all(np.diff(w, axis=1) <= 0)                        # descending, as top-k returns them


def test_layer_routing_structure():
    for name in ("layer_decode_t64", "layer_prefill_t4096"):
        wl = WORKLOADS[name]
        inp = layer_inputs(wl, with_weights=False)
        assert inp["x"].shape == (wl.T, wl.H) and inp["x"].dtype == np.uint16   # bf16 bits
        _check_routing(inp, wl.E, wl.k)
    wl = WORKLOADS["layer_decode_t64"]
    ids = layer_inputs(wl, with_weights=False)["topk_ids"]
    # 64 tokens x 8 slots over 256 experts: about 256 (1 - (1 - 8/256)^64) = 222 experts touched
    assert 200 <= len(np.unique(ids)) <= 240


def test_training_workload_has_a_hot_expert():
    wl = WORKLOADS["layer_train_t16384"]
    inp = layer_inputs(wl, tokens=4096, with_weights=False)
    _check_routing(inp, wl.E, wl.k)
    counts = np.bincount(inp["topk_ids"].ravel(), minlength=wl.E)
    assert counts.max() > 3 * np.median(counts)                   # the +2 logit bias on one expert
