"""Host logic of bench.py, on the CPU: the multi-rank reduction of the timed
region (world size 2 over gloo), the whole-job throughput, the reference arm's
JSON line, and the bookkeeping that feeds the roofline (launch counts, the
source-hash gate on measured DRAM traffic)."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(values[rank], world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    """Each rank timed its own region; every rank ends up with the slowest."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    values = [7.25, 9.5]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, values, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 9.5, 1: 9.5}


def test_single_rank_needs_no_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_job_throughput_counts_every_rank():
    # 16384 tokens a step on each of 4 replicas, the slowest taking 8 ms
    assert bench.job_throughput(16384, 4, 8.0) == pytest.approx(4 * 16384 / 0.008)
    assert bench.job_throughput(16384, 1, 8.0) == pytest.approx(16384 / 0.008)


def test_permute_launch_count():
    assert bench.permute_launches(512) == 2      # one-block index kernel + gather
    assert bench.permute_launches(1024) == 2
    assert bench.permute_launches(1025) == 3     # count, rank, gather
    assert bench.permute_launches(131072) == 3


def test_traffic_is_reported_only_for_the_captured_sources(monkeypatch):
    entry = {"workload": "layer_train_t16384", "bytes_per_launch": 1.0e9, "sources": {"gmm.cu": "0" * 64}}
    monkeypatch.setattr(bench, "GMM_TRAFFIC", [entry])
    assert bench.measured_gmm_traffic("layer_train_t16384") is None     # the hash no longer matches
    assert bench.measured_gmm_traffic("layer_decode_t64") is None       # no capture for this workload
    import hashlib
    with open(os.path.join(ROOT, "moe_routed_expert_gb300", "csrc", "gmm.cu"), "rb") as f:
        entry["sources"]["gmm.cu"] = hashlib.sha256(f.read()).hexdigest()
    assert bench.measured_gmm_traffic("layer_train_t16384") == 1.0e9


def _run_reference(env_extra):
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "gmm_tiny_e4", "--steps", "2", "--warmup", "1"], capture_output=True, text=True,
                       env=env, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout


def test_reference_arm_json_line():
    lines = [l for l in _run_reference({}).splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["steps"] == 2 and d["vs_baseline"] is None
    assert d["config"]["workload"] == "gmm_tiny_e4"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    out = _run_reference({"RANK": "1", "WORLD_SIZE": "2"})
    assert not [l for l in out.splitlines() if l.startswith("{")]


def test_layer_roofline_bytes_of_the_prefill_layer():
    """Weights of every expert with rows once, tokens in and out once, routing once:
    256 live experts x 3 H I bf16 + 2 T H bf16 + T k (int32 + fp32) = 1.644 GB."""
    from workloads import WORKLOADS as W
    wl = W["layer_prefill_t4096"]
    ids = np.tile(np.arange(8, dtype=np.int32), (wl.T, 1))
    ids[:, :] = (np.arange(wl.T * 8).reshape(wl.T, 8) % wl.E).astype(np.int32)   # every expert holds rows
    b = bench.layer_bytes(wl, {"topk_ids": ids})
    assert b == 256 * 3 * 2048 * 512 * 2 + 2 * 4096 * 2048 * 2 + 4096 * 8 * 8
    assert abs(b / 1e9 - 1.644) < 0.001
    ids[:, :] = 0   # one expert: only its weights count
    assert bench.layer_bytes(wl, {"topk_ids": ids}) == 3 * 2048 * 512 * 2 + 2 * 4096 * 2048 * 2 + 4096 * 8 * 8


def test_cpu_baseline_and_reference_arm_share_one_sample():
    """Both CPU arms time the same oracle sample of the same workload."""
    from workloads import WORKLOADS as W, layer_inputs
    wl = W["layer_decode_t64"]
    inp = {"topk_ids": np.zeros((wl.T, wl.k), np.int32), "topk_w": np.zeros((wl.T, wl.k), np.float32),
           "x": np.zeros((wl.T, wl.H), np.uint16)}
    _, units_a, unit_a, desc_a = bench.cpu_sample("layer_decode_t64", inp)
    _, units_b, unit_b, desc_b = bench.cpu_sample("layer_decode_t64", inp)
    assert (units_a, unit_a, desc_a) == (units_b, unit_b, desc_b)
    assert "first 8 of 64 tokens" in desc_a and "experts 0..31 of 256" in desc_a
    assert bench.cpu_model()
    assert bench.cpu_threads() >= 1
