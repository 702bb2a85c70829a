"""Benchmark of the routed-expert MoE hot path on GB300.

Default workload: the MoE layer training step (T=16384 tokens, hidden 4096,
64 experts, top-8, intermediate 1024, SwiGLU clip 7, one hot expert): permute,
gate_up GMM with the SwiGLU epilogue, down GMM, weighted combine, then the
whole backward (combine gradients, dX and dW of both GMMs, SwiGLU gradient,
token gradient).  One step = one forward + backward over one batch.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                        [--extra default|none|mx|all] [--impl reference] [--nvtx]

Prints one JSON line.  ``value`` is tokens/s of the whole job with inputs
resident in HBM, timed with CUDA events on the launching stream between a
barrier + synchronize on both sides (max over ranks); ``e2e`` is the same
metric through the public layer entry points with host (pinned) inputs and
outputs copied inside the timed region.  Under torchrun every rank runs its
own replica (the layer shards by batch with no data-path exchange), so the
scaling is weak.  ``--impl reference`` times the CPU oracle on a bounded
token sample of the same workload.

With the default workload the line also carries ``workloads``: the Zipf
grouped matmul forward + backward (E=8, K=1024, N=2048, M=8192; tensor-bound),
the prefill (T=4096) and decode (T=64) layer forwards (HBM-bound), and the
same layers in A8W4-FP and A4W4-FP (MXFP4 weights), each timed the same way
with its own per-launch split, roofline, clocks and e2e.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from workloads import WORKLOADS, gmm_inputs, layer_inputs, mx_layer_weights, pack_fp4  # noqa: E402

METRIC = "GMM fwd+bwd TFLOP/s and MoE-layer tokens/s on 1 GB300; % of bf16 peak / HBM BW"
DEFAULT_WORKLOAD = "layer_train_t16384"

# DRAM bytes per GMM launch (the mean over one step's GMM launches), each from
# one ncu capture of the sources with these hashes; reported only while they
# match (the captures' commands sit beside their summaries).
GMM_TRAFFIC = [
    {"workload": "layer_train_t16384", "bytes_per_launch": 2.693e9,
     "sources": {"gmm.cu": "4376a8c0af4fe31054a2e34448ac98ffc1291363faa2891dbfc3494167497b5f",
                 "gmm_pair.cu": "7acdcaeb39a20463640220649c863932e342290ca1dae165d40bfcb594943a1f",
                 "common.cuh": "0408a2178e2f80598505925f2d7a91553ba5aefc51b89e8a1bc927e9ee3fbfcd",
                 "sched.cuh": "3e1e8e7b2a17ea21d2a8bff7550b0730d5170eabf1c4d36c95b442e3a7e89365"}},
    {"workload": "layer_prefill_t4096", "bytes_per_launch": 1.836e9,
     "sources": {"gmm.cu": "4376a8c0af4fe31054a2e34448ac98ffc1291363faa2891dbfc3494167497b5f", "common.cuh": "0408a2178e2f80598505925f2d7a91553ba5aefc51b89e8a1bc927e9ee3fbfcd"}},
    {"workload": "layer_decode_t64", "bytes_per_launch": 1.4158e9,
     "sources": {"gmm.cu": "4376a8c0af4fe31054a2e34448ac98ffc1291363faa2891dbfc3494167497b5f", "common.cuh": "0408a2178e2f80598505925f2d7a91553ba5aefc51b89e8a1bc927e9ee3fbfcd"}},
    {"workload": "gmm_zipf_e8", "bytes_per_launch": 7.58e7,
     "sources": {"gmm.cu": "4376a8c0af4fe31054a2e34448ac98ffc1291363faa2891dbfc3494167497b5f",
                 "gmm_pair.cu": "7acdcaeb39a20463640220649c863932e342290ca1dae165d40bfcb594943a1f",
                 "common.cuh": "0408a2178e2f80598505925f2d7a91553ba5aefc51b89e8a1bc927e9ee3fbfcd",
                 "sched.cuh": "3e1e8e7b2a17ea21d2a8bff7550b0730d5170eabf1c4d36c95b442e3a7e89365"}},
    {"workload": "layer_prefill_mx_t4096", "bytes_per_launch": 5.179e8,
     "sources": {"gmm_mx.cu": "72a42ef9d9137faeff13650d3ac3feb3baf11564ae897628e5f19e1c254733cc", "mx.cuh": "8184ef27c720621f7414f59e02aa9014a885853c33cc323bb1750e932d249ffd", "common.cuh": "0408a2178e2f80598505925f2d7a91553ba5aefc51b89e8a1bc927e9ee3fbfcd"}},
    {"workload": "layer_decode_mx_t64", "bytes_per_launch": 3.683e8,
     "sources": {"gmm_mx.cu": "72a42ef9d9137faeff13650d3ac3feb3baf11564ae897628e5f19e1c254733cc", "mx.cuh": "8184ef27c720621f7414f59e02aa9014a885853c33cc323bb1750e932d249ffd", "common.cuh": "0408a2178e2f80598505925f2d7a91553ba5aefc51b89e8a1bc927e9ee3fbfcd"}},
    {"workload": "layer_prefill_a8w4_t4096", "bytes_per_launch": 3.108e8,
     "sources": {"gmm_mx.cu": "72a42ef9d9137faeff13650d3ac3feb3baf11564ae897628e5f19e1c254733cc", "mx.cuh": "8184ef27c720621f7414f59e02aa9014a885853c33cc323bb1750e932d249ffd", "common.cuh": "0408a2178e2f80598505925f2d7a91553ba5aefc51b89e8a1bc927e9ee3fbfcd"}},
    {"workload": "layer_decode_a8w4_t64", "bytes_per_launch": 1.928e8,
     "sources": {"gmm_mx.cu": "72a42ef9d9137faeff13650d3ac3feb3baf11564ae897628e5f19e1c254733cc", "mx.cuh": "8184ef27c720621f7414f59e02aa9014a885853c33cc323bb1750e932d249ffd", "common.cuh": "0408a2178e2f80598505925f2d7a91553ba5aefc51b89e8a1bc927e9ee3fbfcd"}},
    {"workload": "layer_prefill_a4w4_t4096", "bytes_per_launch": 2.927e8,
     "sources": {"gmm_mx.cu": "72a42ef9d9137faeff13650d3ac3feb3baf11564ae897628e5f19e1c254733cc", "mx.cuh": "8184ef27c720621f7414f59e02aa9014a885853c33cc323bb1750e932d249ffd", "common.cuh": "0408a2178e2f80598505925f2d7a91553ba5aefc51b89e8a1bc927e9ee3fbfcd"}},
    {"workload": "layer_decode_a4w4_t64", "bytes_per_launch": 1.926e8,
     "sources": {"gmm_mx.cu": "72a42ef9d9137faeff13650d3ac3feb3baf11564ae897628e5f19e1c254733cc", "mx.cuh": "8184ef27c720621f7414f59e02aa9014a885853c33cc323bb1750e932d249ffd", "common.cuh": "0408a2178e2f80598505925f2d7a91553ba5aefc51b89e8a1bc927e9ee3fbfcd"}},
]


def measured_gmm_traffic(workload):
    import hashlib
    csrc = os.path.join(ROOT, "moe_routed_expert_gb300", "csrc")
    for entry in GMM_TRAFFIC:
        if entry["workload"] != workload:
            continue
        for name, digest in entry["sources"].items():
            with open(os.path.join(csrc, name), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != digest:
                    return None
        return entry["bytes_per_launch"]
    return None


# ---------------------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            out_dir = os.environ.get("MOE_BENCH_CLOCKS_DIR", tempfile.gettempdir())
            os.makedirs(out_dir, exist_ok=True)
            self.path = os.path.join(out_dir, "moe_bench_clocks_rank%d.csv" % self.gpu)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names, r[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        loaded = [r for r in rows if r[2] > 200.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows), "reasons": sorted(reasons)}


def permute_launches(nslots):
    """Kernels one permute launches: a one-block index kernel and the gather up to
    1024 routed slots, else count, rank and the gather."""
    return 2 if nslots <= 1024 else 3


def bf16_dev(bits, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


# ---------------------------------------------------------------------------- GPU steps
class LayerTrainStep:
    """Forward + backward of the routed-expert layer, as the sequence of C-ABI
    calls the layer entry points make (so each GMM launch can be timed)."""

    def __init__(self, wl, dev, inp):
        import torch
        import moe_routed_expert_gb300 as M
        self.M, self.wl, self.dev = M, wl, dev
        T, H, E, k, I = wl.T, wl.H, wl.E, wl.k, wl.I
        R = T * k
        self.x = bf16_dev(inp["x"], dev)
        self.w1 = bf16_dev(inp["w1"], dev)
        self.w2 = bf16_dev(inp["w2"], dev)
        self.dy = bf16_dev(inp["dy"], dev)
        self.ids = torch.from_numpy(inp["topk_ids"]).to(dev)
        self.tw = torch.from_numpy(inp["topk_w"]).to(dev)
        self.saved = M.LayerSaved(T, H, I, E, k, dev)
        bf = torch.bfloat16
        self.y = torch.empty(T, H, dtype=bf, device=dev)
        self.dy2 = torch.empty(R, H, dtype=bf, device=dev)
        self.dh = torch.empty(R, 2 * I, dtype=bf, device=dev)
        self.dx = torch.empty(T, H, dtype=bf, device=dev)
        self.dw1 = torch.empty_like(self.w1)
        self.dw2 = torch.empty_like(self.w2)
        self.dprobs = torch.empty(T, k, dtype=torch.float32, device=dev)
        self.ws = M.Workspace(max(M.moe_permute_workspace_size(T, k, E), M.moe_layer_workspace_size(T, H, I, E, k)),
                              dev)
        gl = inp["topk_ids"]
        counts = np.bincount(gl[gl >= 0].ravel(), minlength=E)
        Rr = int(counts.sum())
        f_up, f_dn = 2.0 * Rr * H * 2 * I, 2.0 * Rr * I * H
        self.stages = [
            ("permute", self.permute, 0.0, permute_launches(T * k)),
            ("gmm_fwd_gate_up_swiglu", self.gmm1, f_up, 1),
            ("gmm_fwd_down", self.gmm2, f_dn, 1),
            ("combine", self.combine, 0.0, 1),
            ("combine_bwd", self.combine_bwd, 0.0, 1),
            ("gmm_dx_down_swiglu_bwd", self.dx_down_swiglu, f_dn, 1),
            ("gmm_dw_down", self.dw_down, f_dn, 1),
            ("gmm_dx_gate_up", self.dx_up, f_up, 1),
            ("gmm_dw_gate_up", self.dw_up, f_up, 1),
            ("permute_bwd", self.permute_bwd, 0.0, 1),
        ]
        self.units = T  # tokens per step
        self.unit = "tokens/s"

    def permute(self):
        s = self.saved
        self.M.moe_permute(self.x, self.ids, self.wl.E, out=(s.x_perm, s.group_list, s.row_id_map, s.sorted_flat),
                           ws=self.ws)

    def gmm1(self):
        s = self.saved
        self.M.gmm_forward(s.x_perm, self.w1, s.group_list, epilogue=1, clip=self.wl.clip, y=s.a, h_save=s.h,
                           ws=self.ws)

    def gmm2(self):
        s = self.saved
        self.M.gmm_forward(s.a, self.w2, s.group_list, y=s.y2, ws=self.ws)

    def combine(self):
        s = self.saved
        self.M.moe_unpermute(s.y2, s.row_id_map, self.tw, self.wl.T, self.wl.k, y=self.y, ws=self.ws)

    def combine_bwd(self):
        s = self.saved
        self.M.moe_unpermute_backward(self.dy, s.y2, s.row_id_map, self.tw, self.wl.k, dy_perm=self.dy2,
                                      dprobs=self.dprobs, ws=self.ws)

    def dx_down_swiglu(self):
        # dH = SwiGLU'(H, dY2 @ W2^T) in one grouped matmul, as the layer backward does
        s = self.saved
        self.M.gmm_backward_dx_swiglu(self.dy2, self.w2, s.group_list, s.h, self.wl.clip, dh=self.dh, ws=self.ws)

    def dw_down(self):
        s = self.saved
        self.M.gmm_backward(s.a, self.w2, s.group_list, self.dy2, need_dx=False, dw=self.dw2, ws=self.ws)

    def dx_up(self):
        s = self.saved
        # dx_perm reuses the dY2 buffer, as the layer entry point does
        self.M.gmm_backward(s.x_perm, self.w1, s.group_list, self.dh, need_dw=False, dx=self.dy2, ws=self.ws)

    def dw_up(self):
        s = self.saved
        self.M.gmm_backward(s.x_perm, self.w1, s.group_list, self.dh, need_dx=False, dw=self.dw1, ws=self.ws)

    def permute_bwd(self):
        self.M.moe_permute_backward(self.dy2, self.saved.row_id_map, self.wl.T, self.wl.k, dx=self.dx, ws=self.ws)

    # public entry points with host buffers, for e2e
    def e2e_host_inputs(self, inp):
        return {"x": pinned_bf16(inp["x"]), "dy": pinned_bf16(inp["dy"]), "topk_ids": pinned(inp["topk_ids"]),
                "topk_w": pinned(inp["topk_w"])}

    def e2e_outputs(self):
        import torch
        T, H, k = self.wl.T, self.wl.H, self.wl.k
        return {"y": torch.empty(T, H, dtype=torch.bfloat16, device=self.dev),
                "dx": torch.empty(T, H, dtype=torch.bfloat16, device=self.dev),
                "dprobs": torch.empty(T, k, dtype=torch.float32, device=self.dev)}

    def e2e_compute(self, i, o):
        M, wl = self.M, self.wl
        M.moe_layer_forward(i["x"], i["topk_ids"], i["topk_w"], self.w1, self.w2, wl.clip, saved=self.saved, y=o["y"],
                            ws=self.ws)
        M.moe_layer_backward(i["dy"], i["topk_w"], self.w1, self.w2, self.saved, wl.clip, dx=o["dx"], dw1=self.dw1,
                             dw2=self.dw2, dprobs=o["dprobs"], ws=self.ws)

    e2e_api = "moe_layer_forward/moe_layer_backward"


fused_combine = False   # --down-combine fused


class LayerFwdStep(LayerTrainStep):
    """Forward only (prefill / decode layer workloads).  Where the layer entry
    point fuses the dispatch into gate_up (inference, groups averaging under
    512 rows), a step is one moe_layer_forward call, and the per-kernel split
    times the same launches through their own entry points: the permute's
    index pass, the gate_up GMM gathering its rows from x, the down GMM and
    the combine."""

    def __init__(self, wl, dev, inp):
        import torch
        inp = dict(inp)
        inp["dy"] = inp["x"]
        super().__init__(wl, dev, inp)
        ids = inp["topk_ids"]
        counts = np.bincount(ids[ids >= 0].ravel(), minlength=wl.E)
        live = int((counts > 0).sum())
        R = int(counts.sum())
        T, H, I, k = wl.T, wl.H, wl.I, wl.k
        self.fused = wl.T * wl.k < 512 * wl.E
        if not self.fused:
            self.stages = self.stages[:4]
            # algorithmic bytes of the GMMs: weights of non-empty experts + activations in/out once
            self.gmm_bytes = {"gmm_fwd_gate_up_swiglu": live * H * 2 * I * 2 + R * H * 2 + R * I * 2,
                              "gmm_fwd_down": live * I * H * 2 + R * I * 2 + R * H * 2}
            return
        M = self.M
        self.y_layer = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        f_up, f_dn = 2.0 * R * H * 2 * I, 2.0 * R * I * H
        self.ws_mlp = M.Workspace(M.moe_expert_mlp_workspace_size(T, k, wl.E), dev)
        self.stages = [
            ("permute_index", self.permute_index, 0.0, permute_launches(T * k) - 1),
            ("gmm_expert_mlp", self.expert_mlp, f_up + f_dn, 1),
            ("combine", self.combine, 0.0, 1),
        ]
        # algorithmic bytes of the one launch of both GMMs: weights of the
        # experts with rows once, the tokens once (gathered k times, from L2),
        # the activation out and back in once, the expert outputs once
        self.gmm_bytes = {"gmm_expert_mlp": live * 3 * H * I * 2 + T * H * 2 + 2 * R * I * 2 + R * H * 2}
        self.headline = self.layer_call
        if fused_combine:
            # the gathered gate_up GMM, then the down GMM fused with the combine
            # (gmm_forward_combine) in place of the one launch and the combine
            self.ws_comb = M.Workspace(M.gmm_forward_combine_workspace_size(T, k, T * k, H), dev)
            self.stages = [self.stages[0], ("gmm_gate_up_gather_act", self.gmm1_gather, f_up, 1),
                           ("gmm_down_combine", self.gmm2_combine, f_dn, 1)]
            self.gmm_bytes = {"gmm_gate_up_gather_act": live * H * 2 * I * 2 + T * H * 2 + R * I * 2,
                              "gmm_down_combine": live * I * H * 2 + R * I * 2 + T * H * 2}
            self.headline = None
        self.kernel = "expert_mlp_kernel (gate_up gathering its rows from the tokens, then down, one launch)"

    def permute_index(self):
        s = self.saved
        self.M.moe_permute(None, self.ids, self.wl.E, out=(None, s.group_list, s.row_id_map, s.sorted_flat),
                           ws=self.ws)

    def gmm1_gather(self):
        s = self.saved
        self.M.gmm_forward_gather_act(self.x, s.sorted_flat, self.wl.k, self.w1, s.group_list, ("swiglu", [self.wl.clip]),
                                      y=s.a, ws=self.ws)


    def expert_mlp(self):
        s = self.saved
        self.M.moe_expert_mlp_forward(self.x, s.sorted_flat, s.group_list, self.w1, self.w2, self.wl.k,
                                      ("swiglu", [self.wl.clip]), a=s.a, y2=s.y2, ws=self.ws_mlp)

    def gmm2_combine(self):
        s = self.saved
        self.M.gmm_forward_combine(s.a, self.w2, s.group_list, s.row_id_map, s.sorted_flat, self.tw, y=self.y,
                                   ws=self.ws_comb)

    def layer_call(self):
        self.M.moe_layer_forward(self.x, self.ids, self.tw, self.w1, self.w2, self.wl.clip, y=self.y_layer,
                                 ws=self.ws)

    def e2e_host_inputs(self, inp):
        return {"x": pinned_bf16(inp["x"]), "topk_ids": pinned(inp["topk_ids"]), "topk_w": pinned(inp["topk_w"])}

    def e2e_outputs(self):
        import torch
        return {"y": torch.empty(self.wl.T, self.wl.H, dtype=torch.bfloat16, device=self.dev)}

    def e2e_compute(self, i, o):
        self.M.moe_layer_forward(i["x"], i["topk_ids"], i["topk_w"], self.w1, self.w2, self.wl.clip, y=o["y"],
                                 ws=self.ws)

    e2e_api = "moe_layer_forward"


class LayerMxStep:
    """The MX layer forward (A8W8-FP, A8W4-FP, A4W4-FP) as the calls
    moe_layer_forward_mx makes: quantising permute, block-scaled gate_up GMM with
    the activation and Q_MX in its epilogue, block-scaled down GMM, combine."""

    def __init__(self, wl, dev, inp):
        import torch
        import moe_routed_expert_gb300 as M
        self.M, self.wl, self.dev = M, wl, dev
        T, H, E, k, I = wl.T, wl.H, wl.E, wl.k, wl.I
        R = T * k
        u8 = torch.uint8
        self.x = bf16_dev(inp["x"], dev)
        self.ids = torch.from_numpy(inp["topk_ids"]).to(dev)
        self.tw = torch.from_numpy(inp["topk_w"]).to(dev)
        self.wfmt = wl.w_mx or wl.mx
        self.afmt = M.activation_format(wl.mx)
        pk = (lambda a: pack_fp4(a)) if self.wfmt == "e2m1" else (lambda a: a)   # E2M1: two codes per byte
        self.w1q, self.w2q = (torch.from_numpy(pk(inp[n])).to(dev) for n in ("w1_q", "w2_q"))
        self.w1s, self.w2s = (torch.from_numpy(inp[n]).to(dev) for n in ("w1_s", "w2_s"))
        xb = 0.5 if wl.mx == "e2m1" else 1.0
        self.xq = torch.empty(R, int(H * xb), dtype=u8, device=dev)
        self.xs = torch.empty(R, H // 32, dtype=u8, device=dev)
        self.gl = torch.empty(E, dtype=torch.int64, device=dev)
        self.rmap = torch.empty(R, dtype=torch.int32, device=dev)
        self.sflat = torch.empty(R, dtype=torch.int32, device=dev)
        self.aq = torch.empty(R, I, dtype=u8, device=dev)
        self.as_ = torch.empty(R, I // 32, dtype=u8, device=dev)
        self.o = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
        self.y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        self.ws = M.Workspace(max(M.moe_permute_workspace_size(T, k, E), M.moe_layer_mx_workspace_size(T, H, I, E, k)),
                              dev)
        self.act = ("swiglu", [wl.clip])
        ids = inp["topk_ids"]
        counts = np.bincount(ids[ids >= 0].ravel(), minlength=E)
        live = int((counts > 0).sum())
        Rr = int(counts.sum())
        f_up, f_dn = 2.0 * Rr * H * 2 * I, 2.0 * Rr * I * H
        self.stages = [
            ("permute_mx", self.permute, 0.0, permute_launches(R)),
            ("gmm_mx_gate_up_act_quant", self.gmm1, f_up, 1),
            ("gmm_mx_down", self.gmm2, f_dn, 1),
            ("combine", self.combine, 0.0, 1),
        ]
        # algorithmic bytes: weights (fp8, or E2M1 at half a byte) and their scales of the
        # non-empty experts, operands in and results out once
        wb = 0.5 if self.wfmt == "e2m1" else 1.0
        self.gmm_bytes = {"gmm_mx_gate_up_act_quant": live * 2 * I * (wb * H + H // 32) + Rr * (xb * H + H // 32)
                          + Rr * (I + I // 32),
                          "gmm_mx_down": live * H * (wb * I + I // 32) + Rr * (I + I // 32) + Rr * H * 2}
        self.units = T
        self.unit = "tokens/s"
        self.dtype = (("mxfp4_" if wl.mx == "e2m1" else "mxfp8_") + wl.mx
                      + ("_w" + self.wfmt if self.wfmt != wl.mx else "")
                      + ("_a" + self.afmt if self.afmt != wl.mx else ""))
        self.kernel = "gmm_mx_kernel (both block-scaled GMM launches of a step)"

    def permute(self):
        self.M.moe_permute_mx(self.x, self.ids, self.wl.E, self.wl.mx,
                              out=(self.xq, self.xs, self.gl, self.rmap, self.sflat), ws=self.ws)

    def gmm1(self):
        self.M.gmm_forward_mx(self.xq, self.xs, self.w1q, self.w1s, self.gl, x_fmt=self.wl.mx, w_fmt=self.wfmt,
                              activation=self.act, a_q=self.aq, a_scales=self.as_, ws=self.ws)

    def gmm2(self):
        self.M.gmm_forward_mx(self.aq, self.as_, self.w2q, self.w2s, self.gl, x_fmt=self.afmt, w_fmt=self.wfmt,
                              y=self.o, ws=self.ws)

    def combine(self):
        self.M.moe_unpermute(self.o, self.rmap, self.tw, self.wl.T, self.wl.k, y=self.y, ws=self.ws)

    def e2e_host_inputs(self, inp):
        return {"x": pinned_bf16(inp["x"]), "topk_ids": pinned(inp["topk_ids"]), "topk_w": pinned(inp["topk_w"])}

    def e2e_outputs(self):
        import torch
        return {"y": torch.empty(self.wl.T, self.wl.H, dtype=torch.bfloat16, device=self.dev)}

    def e2e_compute(self, i, o):
        self.M.moe_layer_forward_mx(i["x"], i["topk_ids"], i["topk_w"], self.w1q, self.w1s, self.w2q, self.w2s,
                                    x_fmt=self.wl.mx, w_fmt=self.wfmt, activation=self.act, y=o["y"], ws=self.ws)

    e2e_api = "moe_layer_forward_mx"


class GmmStep:
    """Standalone grouped matmul forward + dX + dW (the Zipf GMM workload).

    Its inputs (x 16.8 MB, W 33.5 MB, dY 33.5 MB) fit in L2, so the steps
    rotate through ``nsets`` copies of every input and output: a step reads
    inputs last touched ``nsets`` steps earlier, with more than L2's capacity
    of other traffic in between."""

    def __init__(self, wl, dev, inp, nsets=1):
        import torch
        import moe_routed_expert_gb300 as M
        self.M, self.wl, self.dev = M, wl, dev
        self.sets = []
        for _ in range(nsets):
            b = {"x": bf16_dev(inp["x"], dev), "w": bf16_dev(inp["w"], dev),
                 "dy": bf16_dev(inp["dy"], dev) if "dy" in inp else None,
                 "gl": torch.from_numpy(inp["group_list"]).to(dev),
                 "y": torch.empty(wl.M, wl.N, dtype=torch.bfloat16, device=dev)}
            b["dx"] = torch.empty_like(b["x"])
            b["dw"] = torch.empty_like(b["w"])
            self.sets.append(b)
        self.cur = self.sets[0]
        self.nstep = 0
        # the e2e leg keeps the weights of set 0 resident and copies x and dY in
        self.w, self.gl, self.y, self.dx, self.dw = (self.cur[n] for n in ("w", "gl", "y", "dx", "dw"))
        self.ws = M.Workspace(256, dev)
        f = 2.0 * wl.M * wl.K * wl.N
        self.stages = [("gmm_fwd", self.fwd, f, 1)]
        if wl.backward:
            # one gmm_backward call: dX and dW (one CTA-pair launch, or two side by side)
            self.stages += [("gmm_bwd_dx_dw", self.bwd, 2 * f, 2)]
        self.units = sum(s[2] for s in self.stages) / 1e12
        self.unit = "TFLOP/s"
        set_bytes = sum(t.numel() * t.element_size() for t in self.sets[0].values() if t is not None)
        self.l2 = ("%d rotating sets of inputs and outputs (%.0f MB each), more than L2 between reuses"
                   % (nsets, set_bytes / 1e6)) if nsets > 1 else "inputs smaller than L2, not rotated"

    def advance(self):
        self.cur = self.sets[self.nstep % len(self.sets)]
        self.nstep += 1

    def fwd(self):
        c = self.cur
        self.M.gmm_forward(c["x"], c["w"], c["gl"], y=c["y"], ws=self.ws)

    def bwd(self):
        c = self.cur
        self.M.gmm_backward(c["x"], c["w"], c["gl"], c["dy"], dx=c["dx"], dw=c["dw"], ws=self.ws)

    def e2e_host_inputs(self, inp):
        return {"x": pinned_bf16(inp["x"]), "dy": pinned_bf16(inp["dy"])}

    def e2e_outputs(self):
        import torch
        return {"y": torch.empty_like(self.y), "dx": torch.empty_like(self.dx)}

    def e2e_compute(self, i, o):
        self.M.gmm_forward(i["x"], self.w, self.gl, y=o["y"], ws=self.ws)
        self.M.gmm_backward(i["x"], self.w, self.gl, i["dy"], dx=o["dx"], dw=self.dw, ws=self.ws)

    e2e_api = "gmm_forward/gmm_backward"


def pinned(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def pinned_bf16(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).pin_memory()


class E2EPipeline:
    """Every step copies its inputs host->device and its results device->host
    (pinned buffers).  Two buffer sets let the copies of neighbouring steps run
    on their own streams while a step computes; each step still waits for its
    own inputs, and the timed region ends when the last results are on the host."""

    def __init__(self, step, inp, nbuf=2):
        import torch
        self.step, self.nbuf = step, nbuf
        self.h_in = step.e2e_host_inputs(inp)
        self.d_in = [{k: torch.empty(v.shape, dtype=v.dtype, device=step.dev) for k, v in self.h_in.items()}
                     for _ in range(nbuf)]
        self.d_out = [step.e2e_outputs() for _ in range(nbuf)]
        self.h_out = [{k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in d.items()} for d in self.d_out]
        self.h2d = torch.cuda.Stream(device=step.dev)
        self.d2h = torch.cuda.Stream(device=step.dev)
        ev = lambda: [torch.cuda.Event() for _ in range(nbuf)]
        self.in_ready, self.in_free, self.done, self.out_free = ev(), ev(), ev(), ev()
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in self.h_in.values())
        self.d2h_bytes = sum(t.numel() * t.element_size() for t in self.h_out[0].values())

    def run(self, steps):
        import torch
        comp = torch.cuda.current_stream()
        for i in range(steps):
            b = i % self.nbuf
            self.h2d.wait_event(self.in_free[b])
            with torch.cuda.stream(self.h2d):
                for k, v in self.h_in.items():
                    self.d_in[b][k].copy_(v, non_blocking=True)
            self.in_ready[b].record(self.h2d)
            comp.wait_event(self.in_ready[b])
            comp.wait_event(self.out_free[b])
            self.step.e2e_compute(self.d_in[b], self.d_out[b])
            self.in_free[b].record(comp)
            self.done[b].record(comp)
            self.d2h.wait_event(self.done[b])
            with torch.cuda.stream(self.d2h):
                for k, v in self.d_out[b].items():
                    self.h_out[b][k].copy_(v, non_blocking=True)
            self.out_free[b].record(self.d2h)
        for b in range(self.nbuf):
            comp.wait_event(self.out_free[b])


def make_step(name, dev, tokens=None, nsets=1):
    wl = WORKLOADS[name]
    if name.startswith("gmm"):
        inp = gmm_inputs(wl)
        return GmmStep(wl, dev, inp, nsets=nsets), inp
    if wl.mx:
        inp = layer_inputs(wl, tokens=tokens, with_weights=False)
        inp.update(mx_layer_weights(wl))
        if tokens is not None:
            wl = wl.with_tokens(tokens)
        return LayerMxStep(wl, dev, inp), inp
    inp = layer_inputs(wl, tokens=tokens)
    if tokens is not None:   # a smaller batch of the same workload (profiling captures)
        wl = wl.with_tokens(tokens)
    return (LayerTrainStep(wl, dev, inp) if wl.backward else LayerFwdStep(wl, dev, inp)), inp


def layer_bytes(wl, inp):
    """Algorithmic HBM bytes of one layer forward (the roofline's numerator):
    the weights of every expert that holds a row, read once, plus the tokens,
    the routing (ids and weights) and the output, once each.  MX weights count
    their codes (E2M1 at half a byte) and E8M0 scales."""
    ids = inp["topk_ids"]
    counts = np.bincount(ids[ids >= 0].ravel(), minlength=wl.E)
    live = int((counts > 0).sum())
    T, H, I, k = wl.T, wl.H, wl.I, wl.k
    if wl.mx:
        wb = 0.5 if (wl.w_mx or wl.mx) == "e2m1" else 1.0
        w = live * (2 * I * (wb * H + H // 32) + H * (wb * I + I // 32))
    else:
        w = live * 3 * H * I * 2
    return w + T * H * 2 * 2 + T * k * 8


# The workloads the default run measures beside its headline: the standalone
# Zipf GMM forward + backward (tensor-bound), the prefill and decode layer
# forwards (HBM-bound), and the same layers with MXFP4 (E2M1) weights and
# MXFP8 or MXFP4 tokens, each with its own split, roofline, clocks and e2e.
EXTRA_WORKLOADS = ["gmm_zipf_e8", "layer_prefill_t4096", "layer_decode_t64", "layer_prefill_a8w4_t4096",
                   "layer_decode_a8w4_t64", "layer_prefill_a4w4_t4096", "layer_decode_a4w4_t64"]
MX_WORKLOADS = ["layer_prefill_mx_t4096", "layer_decode_mx_t64", "layer_prefill_a8w4_t4096",
                "layer_decode_a8w4_t64", "layer_prefill_a4w4_t4096", "layer_decode_a4w4_t64"]
GMM_SETS = 4            # rotating input sets of the Zipf GMM (4 x 168 MB)
MIN_TIMED_MS = 200.0    # the extra workloads run at least this long in their timed region


# ---------------------------------------------------------------------------- CPU oracle (baseline / reference arm)
def oracle_layer_step(wl, inp_sub):
    import oracle as O
    f = O.bf16_bits_to_f64
    x, w1, w2 = f(inp_sub["x"]), f(inp_sub["w1"]), f(inp_sub["w2"])
    y, sv = O.moe_layer_forward(x, inp_sub["topk_ids"], inp_sub["topk_w"], w1, w2, wl.clip)
    if wl.backward:
        O.moe_layer_backward(f(inp_sub["dy"]), sv, inp_sub["topk_w"], w1, w2, wl.clip)


def oracle_mx_layer_step(wl, inp_sub):
    import oracle as O
    from oracle import mx_oracle as X
    X.mx_layer_forward(O.bf16_bits_to_f64(inp_sub["x"]), inp_sub["topk_ids"], inp_sub["topk_w"], inp_sub["w1_q"],
                       inp_sub["w1_s"], inp_sub["w2_q"], inp_sub["w2_s"], wl.mx, wl.w_mx or wl.mx,
                       O.activation("swiglu", [wl.clip]))


def layer_sample(inp, T, E):
    """The first T tokens, with only the slots routed to experts 0..E-1 kept (the
    rest marked unused) and only those experts' weights: every kept expert does
    exactly the work it does in the full problem over those tokens."""
    d = {}
    ids = np.ascontiguousarray(inp["topk_ids"][:T]).copy()
    ids[ids >= E] = -1
    d["topk_ids"] = ids
    for key in ("x", "topk_w", "dy"):
        if key in inp:
            d[key] = np.ascontiguousarray(inp[key][:T])
    for key in ("w1", "w2", "w1_q", "w1_s", "w2_q", "w2_s"):
        if key in inp:
            d[key] = inp[key][:E]
    return d, int((ids >= 0).sum())


def oracle_gmm_step(wl, inp, rows):
    import oracle as O
    f = O.bf16_bits_to_f64
    gl = inp["group_list"].copy()
    # keep the first `rows` rows: trim the groups from the end
    left = rows
    for e in range(len(gl)):
        take = min(gl[e], left)
        gl[e] = take
        left -= take
    x, w = f(inp["x"][:rows]), f(inp["w"])
    O.gmm_forward(x, w, gl)
    if wl.backward:
        O.gmm_backward(x, w, gl, f(inp["dy"][:rows]))


def cpu_sample(name, inp):
    """The oracle's bounded sample of a workload, the same one for the bench's
    cpu_baseline leg and for the reference arm: the first eighth of the tokens
    with the slots and weights of the first eighth of the experts (every kept
    expert does its full-problem work over those tokens), or the first 1024
    rows of a grouped matmul.  Returns (runner, units per run, unit, description)."""
    wl = WORKLOADS[name]
    if name.startswith("gmm"):
        per_row = (3 if wl.backward else 1) * 2.0 * wl.K * wl.N / 1e12
        rows = min(wl.M, 1024)
        desc = "first %d of %d rows (groups trimmed from the end), fwd%s in float64" % (
            rows, wl.M, "+dX+dW" if wl.backward else "")
        return (lambda: oracle_gmm_step(wl, inp, rows)), rows * per_row, "TFLOP/s", desc
    E_s = max(1, wl.E // 8)
    T_s = max(1, wl.T // 8)
    run = oracle_mx_layer_step if wl.mx else oracle_layer_step
    sub, rows = layer_sample(inp, T_s, E_s)
    tok_eq = rows / wl.k   # token-equivalents: a token owns k routed rows
    desc = ("first %d of %d tokens, slots of experts 0..%d of %d kept (%d routed rows = %.0f token-equivalents "
            "at k=%d), layer fwd%s%s in float64" % (T_s, wl.T, E_s - 1, wl.E, rows, tok_eq, wl.k,
                                                    "+bwd" if wl.backward else "",
                                                    " (MX tokens %s, weights %s, quantisation included)"
                                                    % (wl.mx, wl.w_mx or wl.mx) if wl.mx else ""))
    return (lambda: run(wl, sub)), tok_eq, "tokens/s", desc


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.machine()


def cpu_threads():
    """Threads the oracle's numpy/BLAS calls use (OMP/OpenBLAS limits, else every core)."""
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS"):
        v = os.environ.get(var, "")
        if v.isdigit() and int(v) > 0:
            return int(v)
    return os.cpu_count()


def time_cpu_sample(name, inp, runs=None, min_s=10.0, max_runs=8):
    """Time the oracle sample: `runs` runs, or repeat until min_s (at most max_runs).
    Returns (value, unit, sample, seconds, runs)."""
    fn, units, unit, desc = cpu_sample(name, inp)
    times = []
    while True:
        t0 = time.perf_counter()
        fn()
        times.append(time.perf_counter() - t0)
        if runs is not None:
            if len(times) >= runs:
                break
        elif sum(times) >= min_s or len(times) >= max_runs:
            break
    total = sum(times)
    return units * len(times) / total, unit, desc, total, len(times)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    name = args.workload
    wl = WORKLOADS[name]
    if name.startswith("gmm"):
        inp = gmm_inputs(wl)
    elif wl.mx:
        inp = layer_inputs(wl, with_weights=False)
        inp.update(mx_layer_weights(wl))
    else:
        inp = layer_inputs(wl)
    # each step runs the same bounded sample the cpu_baseline leg times
    fn, units, unit, sample = cpu_sample(name, inp)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        fn()
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    v = units * len(times) / total
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": name, "sample": sample},
            "cpu_baseline": {"value": v, "unit": unit, "cores": cpu_threads(), "cpu": cpu_model(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def max_over_ranks(x, world, device=None):
    """The largest of every rank's x: the job ends when its slowest rank does
    (all ranks call it; NCCL on the GPU, any backend the group was made with)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step, world, ms_per_step):
    """Whole-job throughput: the units all ranks processed in a step (replicas,
    each with the same work) over the slowest rank's step time."""
    return units_per_rank_step * world / (ms_per_step / 1e3)


def l2_note(name, step):
    if hasattr(step, "l2"):
        return step.l2
    wl = step.wl
    if name.startswith("layer_decode"):
        return "weights (%s touched) larger than L2" % (
            "0.35 GB" if wl.w_mx == "e2m1" else ("0.7 GB" if wl.mx else "1.4 GB"))
    return "inputs larger than L2"


# ---------------------------------------------------------------------------- one workload on the GPU
def measure(name, step, inp, args, steps, warmup, world, dev, peaks, with_e2e=True):
    """Time `steps` steps of one workload (after `warmup`), then the same steps
    again with an event after every launch for the per-kernel split, then
    (with_e2e) the e2e pipeline.  Returns the workload's JSON fields."""
    import torch
    import moe_routed_expert_gb300 as M
    stream = torch.cuda.current_stream()
    advance = getattr(step, "advance", lambda: None)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    def check():
        st = M.read_status(step.ws)
        assert st == 0, "device status %s" % M.status_string(st)

    # a step: the workload's public call when it has one (the fused layer
    # forward), else its stages in order
    headline = getattr(step, "headline", None)
    run_step = ((lambda: (advance(), headline())) if headline is not None else
                (lambda: (advance(), [fn() for _, fn, _, _ in step.stages])))
    if args.nvtx:   # one range per step around the library's own per-call ranges
        plain_step = run_step

        def run_step():
            torch.cuda.nvtx.range_push("%s step" % name)
            plain_step()
            torch.cuda.nvtx.range_pop()
    # the sampler starts before the warm-up: nvidia-smi's start-up must not land in the timed region
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    for _ in range(warmup):
        run_step()
    check()

    # The headline region records events only at its two ends: an event between
    # two launches would stop the second one's prologue from overlapping the
    # first one's tail (programmatic dependent launch).
    barrier()
    if args.graph:
        # one step captured into a CUDA graph (every call is stream-ordered, with no host
        # synchronisation and no allocation), replayed on the timed stream
        graph = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream(device=dev)
        cs.wait_stream(stream)
        with torch.cuda.stream(cs):
            with torch.cuda.graph(graph, stream=cs):
                headline() if headline is not None else [fn() for _, fn, _, _ in step.stages]
        stream.wait_stream(cs)
        graph.replay()
        barrier()
        check()
        run_step = graph.replay
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(steps):
        run_step()
    t_end.record(stream)
    barrier()
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    check()

    # Per-kernel breakdown: the same steps again with an event after every launch.
    ns = len(step.stages)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(ns + 1)] for _ in range(steps)]
    barrier()
    for s in range(steps):
        ev = events[s]
        advance()
        ev[0].record(stream)
        for i, (sname, fn, _, _) in enumerate(step.stages):
            if args.nvtx:
                torch.cuda.nvtx.range_push(sname)
            fn()
            if args.nvtx:
                torch.cuda.nvtx.range_pop()
            ev[i + 1].record(stream)
    barrier()
    clock_info = clocks.stop()
    check()

    stage_ms = [0.0] * ns
    for s in range(steps):
        for i in range(ns):
            stage_ms[i] += events[s][i].elapsed_time(events[s][i + 1])
    stage_ms = [v / steps for v in stage_ms]
    ms_per_step = elapsed_ms / steps
    value = job_throughput(step.units, world, ms_per_step)

    kernels = {}
    gmm_flops, gmm_ms, gmm_launches = 0.0, 0.0, 0
    launches = 0
    for (sname, _, flops, nl), ms in zip(step.stages, stage_ms):
        entry = {"ms": round(ms, 4), "launches": nl}
        if flops:
            entry["tflops"] = round(flops / (ms / 1e3) / 1e12, 1)
            gmm_flops += flops
            gmm_ms += ms
            gmm_launches += nl
        if hasattr(step, "gmm_bytes") and sname in step.gmm_bytes:
            entry["gbs"] = round(step.gmm_bytes[sname] / (ms / 1e3) / 1e9, 1)
        launches += nl
        kernels[sname] = entry

    if hasattr(step, "gmm_bytes"):
        gbytes = sum(step.gmm_bytes.values())
        achieved = gbytes / (gmm_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": measured_gmm_traffic(name) if args.tokens is None else None,
                "kernel": getattr(step, "kernel", "gmm_kernel (all GMM launches of a step)"),
                "peak_kind": "hbm copy, %s" % peaks["source"]}
    else:
        # every launch of a step that is all grouped matmuls (the standalone
        # GMM workload) runs inside the step's own timed region, where the
        # launches overlap their neighbours' prologues; an event between two
        # launches would stop that, so the step time is the launches' time
        gmm_only = all(flops > 0 for _, _, flops, _ in step.stages)
        achieved = gmm_flops / ((ms_per_step if gmm_only else gmm_ms) / 1e3) / 1e12
        long_step = ms_per_step * steps > 500.0
        peak = peaks["bf16_tflops_sustained"] if long_step else peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4),
                # also against the sustained (power-capped, seconds-long) cuBLAS rate
                "frac_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                "traffic": measured_gmm_traffic(name) if args.tokens is None else None,
                "kernel": "gmm_pair_kernel / gmm_kernel (all %d GMM launches of a step)" % gmm_launches,
                "timing": "the step's timed region (every launch is a GMM)" if gmm_only else
                          "CUDA events around each GMM launch",
                "peak_kind": "bf16 dense %s, %s" % ("sustained" if long_step else "burst", peaks["source"])}

    out = {"value": round(value, 3), "unit": step.unit, "steps": steps, "warmup": warmup,
           "ms_per_step": round(ms_per_step, 4), "dtype": getattr(step, "dtype", "bf16"),
           "config": {"workload": name, **{k_: v_ for k_, v_ in vars(step.wl).items() if k_ != "name"},
                      "l2": l2_note(name, step), "parallelism": "replicas" if world > 1 else "1 GPU"},
           "roofline": roof, "kernels": kernels,
           "launch": "one CUDA graph per step (replayed)" if args.graph else "stream launches, programmatic serialisation",
           "kernels_timing": "CUDA events after every launch, in a second pass of the same steps",
           "gpu_launches": launches * steps,
           "gmm_tflops": round(gmm_flops / (gmm_ms / 1e3) / 1e12, 1) if gmm_ms else None}
    if not name.startswith("gmm") and not getattr(step.wl, "backward", False):
        lb = layer_bytes(step.wl, inp)
        t_roof = lb / (peaks["hbm_gbs"] * 1e9) * 1e3
        out["layer_roofline"] = {"bound": "hbm", "bytes": int(lb), "time_ms": round(t_roof, 4),
                                 "achieved": round(lb / (ms_per_step / 1e3) / 1e9, 1), "peak": peaks["hbm_gbs"],
                                 "unit": "GB/s", "frac": round(t_roof / ms_per_step, 4),
                                 "what": "whole layer step: weights of the experts with rows, tokens, routing and "
                                         "output once each, against the measured copy rate"}
    if clock_info is not None:
        out["clocks"] = clock_info

    # end to end through the public entry points, host buffers, copies inside the timed region
    if with_e2e:
        pipe = E2EPipeline(step, inp)
        pipe.run(2)
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        pipe.h2d.wait_stream(stream)
        pipe.d2h.wait_stream(stream)
        pipe.run(steps)
        b.record(stream)
        barrier()
        e_ms = max_over_ranks(a.elapsed_time(b), world, dev)
        out["e2e"] = {"value": round(job_throughput(step.units, world, e_ms / steps), 3), "unit": step.unit,
                      "h2d_bytes_per_step": int(pipe.h2d_bytes), "d2h_bytes_per_step": int(pipe.d2h_bytes),
                      "ms_per_step": round(e_ms / steps, 4), "api": step.e2e_api,
                      "copies": "pinned host buffers; two buffer sets, H2D and D2H on their own streams"}
        check()
        del pipe
    return out


def extra_steps(step, args, world, dev):
    """Steps for an extra workload: the headline's count, or more, so that its
    timed region lasts at least MIN_TIMED_MS (clock samples land inside it)."""
    import torch
    advance = getattr(step, "advance", lambda: None)
    for _ in range(2):
        advance()
        [fn() for _, fn, _, _ in step.stages]
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(3):
        advance()
        [fn() for _, fn, _, _ in step.stages]
    b.record()
    torch.cuda.synchronize()
    est = max(a.elapsed_time(b) / 3, 1e-3)
    n = max(args.steps, int(np.ceil(MIN_TIMED_MS / est)))
    return int(max_over_ranks(n, world, dev))


# ---------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--extra", default="default", choices=["default", "none", "mx", "all"],
                    help="workloads timed beside the headline: the Zipf GMM and the prefill / decode layers "
                         "(default, with the default workload), none, the MX layers, or all of them")
    ap.add_argument("--nvtx", action="store_true",
                    help="NVTX ranges around each step and each stage of the per-launch split (every call "
                         "of the library is also its own range)")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of one step captured in a CUDA graph (the per-kernel split stays eager)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="run the first T tokens of the layer workload (smaller captures; not a bench line)")
    ap.add_argument("--down-combine", default="split", choices=["split", "fused"],
                    help="layer forwards: the down GMM and the combine as two calls (the layer entry point's "
                         "choice), or the fused gmm_forward_combine")
    args = ap.parse_args()
    global fused_combine
    fused_combine = args.down_combine == "fused"
    if args.impl == "reference":
        return run_reference(args)
    if args.warmup < 3:
        args.warmup = 3

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()

    peaks = load_peaks()
    nsets = GMM_SETS if args.workload.startswith("gmm") and WORKLOADS[args.workload].M >= 1024 else 1
    step, inp = make_step(args.workload, dev, args.tokens, nsets=nsets)
    res = measure(args.workload, step, inp, args, args.steps, args.warmup, world, dev, peaks,
                  with_e2e=not args.no_e2e)
    line = {"metric": METRIC, "value": res["value"], "unit": res["unit"], "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": res["dtype"], "data": "synthetic"}
    line.update({k_: v_ for k_, v_ in res.items() if k_ not in line and k_ not in ("steps", "warmup")})
    if args.tokens is not None:
        line["config"]["note"] = "first %d tokens only: a profiling run, not the workload's bench line" % args.tokens
    if rank == 0 and not args.no_cpu_baseline:
        v, unit, sample, secs, runs = time_cpu_sample(args.workload, inp)
        line["cpu_baseline"] = {"value": round(v, 4), "unit": unit, "cores": cpu_threads(), "cpu": cpu_model(),
                                "kind": "oracle", "sample": sample, "runs": runs, "seconds": round(secs, 2)}

    extras = []
    if args.tokens is None and not args.graph:
        if args.extra in ("default", "all") and (args.workload == DEFAULT_WORKLOAD or args.extra == "all"):
            extras += [w for w in EXTRA_WORKLOADS if w != args.workload]
        if args.extra in ("mx", "all"):
            extras += [w for w in MX_WORKLOADS if w != args.workload and w not in extras]
    if extras:
        del step, inp
        torch.cuda.empty_cache()
        line["workloads"] = {}
        for name in extras:
            nsets = GMM_SETS if name.startswith("gmm") else 1
            st, ip = make_step(name, dev, nsets=nsets)
            n = extra_steps(st, args, world, dev)
            line["workloads"][name] = measure(name, st, ip, args, n, args.warmup, world, dev, peaks,
                                              with_e2e=not args.no_e2e)
            del st, ip
            torch.cuda.empty_cache()
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
