"""Seeded synthetic inputs for the routed-expert MoE hot path.

This module only draws random numbers and lays them out; it holds none of the
hot path's arithmetic.  Both the CPU oracle (``oracle/``) and the CUDA path read
the same bits from here, so a parity test compares two computations on
identical inputs.

Conventions
-----------
* bf16 tensors are returned as ``numpy.uint16`` arrays of raw bfloat16 bits.
  Values are drawn in float32 and rounded to bfloat16 once (round to nearest
  even, through torch's CPU conversion).
* Routing follows the shape of a top-k router: logits ~ N(0, 1) of shape
  [T, E] (one seeded "hot" expert gets a +bias when asked), softmax, top-k in
  descending probability, then the k weights are renormalised to sum to 1.
  Expert ids are int32, weights float32.
* ``group_list`` holds per-expert row counts (int64), not a cumulative sum.
* Every generator takes a seed; a workload's seed is fixed in ``WORKLOADS``.
  numpy's PCG64 ``default_rng`` is used for every draw.

Workloads (sizes of the grouped matmul and MoE layer cases):

=======================  ====================================================
name                     shape
=======================  ====================================================
gmm_tiny_e4              GMM fwd, E=4, K=128, N=256, M=64, expert 2 empty
gmm_zipf_e8              GMM fwd+bwd, E=8, K=1024, N=2048, M=8192, Zipf(1.2)
                         counts over 6 experts, 2 experts empty
layer_prefill_t4096      MoE layer fwd, T=4096, H=2048, E=256, k=8, I=512
layer_decode_t64         MoE layer fwd, T=64, H=2048, E=256, k=8, I=512
layer_train_t16384       MoE layer fwd+bwd, T=16384, H=4096, E=64, k=8,
                         I=1024, SwiGLU clip 7, one hot expert (+2 logit)
layer_prefill_mx_t4096   the prefill layer in MXFP8 (E4M3 tokens and weights)
layer_decode_mx_t64      the decode layer in MXFP8 (E4M3 tokens and weights)
layer_prefill_a8w4_t4096 the prefill layer with E4M3 tokens, MXFP4 (E2M1)
                         weights
layer_decode_a8w4_t64    the decode layer with E4M3 tokens, MXFP4 weights
layer_prefill_a4w4_t4096 the prefill layer with MXFP4 tokens and weights
                         (E4M3 activation)
layer_decode_a4w4_t64    the decode layer with MXFP4 tokens and weights
=======================  ====================================================

MXFP8 weights are drawn directly as codes: N(0, 16^2) draws cast to the fp8
type by torch's CPU conversion (a library cast, not the method's Q_MX), with
E8M0 scale codes drawn uniformly from three values centred so that the
dequantised weights have a standard deviation near 1/sqrt(K).  MXFP4 weights
are codes drawn uniformly from the 16 E2M1 codes (values up to +-6), with
scales centred the same way; the CUDA path takes them packed two per byte,
element 2i in the low nibble (pack_fp4).
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional

import numpy as np

__all__ = [
    "GmmWorkload", "LayerWorkload", "WORKLOADS", "f32_to_bf16_bits",
    "gmm_inputs", "layer_inputs", "routing", "zipf_counts", "normal_bf16",
    "fp8_codes", "e8m0_codes", "mx_weight", "mx_layer_weights", "pack_fp4",
]


@dataclass(frozen=True)
class GmmWorkload:
    name: str
    seed: int
    E: int
    K: int
    N: int
    M: int
    backward: bool
    counts: str  # "tiny" (multinomial over 3 experts, expert 2 empty) or "zipf"

    def flops(self, counts=None) -> float:
        """2*M*K*N per pass (empty groups contribute no rows)."""
        passes = 3 if self.backward else 1
        return passes * 2.0 * self.M * self.K * self.N


@dataclass(frozen=True)
class LayerWorkload:
    name: str
    seed: int
    T: int
    H: int
    E: int
    k: int
    I: int
    clip: float
    hot_bias: float
    backward: bool
    mx: str = ""   # "" (bf16 path) or the tokens' element type in the MX forward
    w_mx: str = ""  # the weights' element type when it differs from mx ("e2m1": MXFP4)

    @property
    def R(self) -> int:
        return self.T * self.k

    def with_tokens(self, T: int) -> "LayerWorkload":
        return replace(self, T=T)


WORKLOADS = {
    "gmm_tiny_e4": GmmWorkload("gmm_tiny_e4", 1, E=4, K=128, N=256, M=64, backward=False, counts="tiny"),
    "gmm_zipf_e8": GmmWorkload("gmm_zipf_e8", 2, E=8, K=1024, N=2048, M=8192, backward=True, counts="zipf"),
    "layer_prefill_t4096": LayerWorkload("layer_prefill_t4096", 3, T=4096, H=2048, E=256, k=8, I=512,
                                         clip=0.0, hot_bias=0.0, backward=False),
    "layer_decode_t64": LayerWorkload("layer_decode_t64", 4, T=64, H=2048, E=256, k=8, I=512,
                                      clip=0.0, hot_bias=0.0, backward=False),
    "layer_train_t16384": LayerWorkload("layer_train_t16384", 5, T=16384, H=4096, E=64, k=8, I=1024,
                                        clip=7.0, hot_bias=2.0, backward=True),
    "layer_prefill_mx_t4096": LayerWorkload("layer_prefill_mx_t4096", 3, T=4096, H=2048, E=256, k=8, I=512,
                                            clip=0.0, hot_bias=0.0, backward=False, mx="e4m3"),
    "layer_decode_mx_t64": LayerWorkload("layer_decode_mx_t64", 4, T=64, H=2048, E=256, k=8, I=512,
                                         clip=0.0, hot_bias=0.0, backward=False, mx="e4m3"),
    "layer_prefill_a8w4_t4096": LayerWorkload("layer_prefill_a8w4_t4096", 3, T=4096, H=2048, E=256, k=8, I=512,
                                              clip=0.0, hot_bias=0.0, backward=False, mx="e4m3", w_mx="e2m1"),
    "layer_decode_a8w4_t64": LayerWorkload("layer_decode_a8w4_t64", 4, T=64, H=2048, E=256, k=8, I=512,
                                           clip=0.0, hot_bias=0.0, backward=False, mx="e4m3", w_mx="e2m1"),
    "layer_prefill_a4w4_t4096": LayerWorkload("layer_prefill_a4w4_t4096", 3, T=4096, H=2048, E=256, k=8, I=512,
                                              clip=0.0, hot_bias=0.0, backward=False, mx="e2m1", w_mx="e2m1"),
    "layer_decode_a4w4_t64": LayerWorkload("layer_decode_a4w4_t64", 4, T=64, H=2048, E=256, k=8, I=512,
                                           clip=0.0, hot_bias=0.0, backward=False, mx="e2m1", w_mx="e2m1"),
}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> raw bfloat16 bits (uint16), round to nearest even (torch CPU cast)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) draws rounded to bfloat16 bits."""
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return f32_to_bf16_bits(a)


def zipf_counts(rng: np.random.Generator, E: int, M: int, n_empty: int, s: float) -> np.ndarray:
    """Counts for E experts summing to M: n_empty experts (seeded choice) get 0 rows,
    the others get shares proportional to r^-s for r = 1.. in a seeded order,
    rounded by largest remainder."""
    perm = rng.permutation(E)
    empty, full = perm[:n_empty], perm[n_empty:]
    r = np.arange(1, len(full) + 1, dtype=np.float64)
    share = r ** (-s)
    share /= share.sum()
    exact = share * M
    base = np.floor(exact).astype(np.int64)
    left = M - int(base.sum())
    order = np.argsort(-(exact - base), kind="stable")
    base[order[:left]] += 1
    counts = np.zeros(E, np.int64)
    counts[full] = base
    counts[empty] = 0
    return counts


def tiny_counts(rng: np.random.Generator, E: int, M: int, empty: int = 2) -> np.ndarray:
    """M rows spread uniformly (multinomial) over every expert but ``empty``."""
    live = [e for e in range(E) if e != empty]
    draw = rng.multinomial(M, [1.0 / len(live)] * len(live))
    counts = np.zeros(E, np.int64)
    counts[live] = draw
    return counts


def gmm_inputs(wl: GmmWorkload, seed: Optional[int] = None) -> dict:
    """x[M,K], w[E,K,N] (bf16 bits), group_list[E] int64 counts, and dy[M,N] when backward."""
    rng = np.random.default_rng(wl.seed if seed is None else seed)
    if wl.counts == "tiny":
        counts = tiny_counts(rng, wl.E, wl.M)
    else:
        counts = zipf_counts(rng, wl.E, wl.M, n_empty=2, s=1.2)
    out = {
        "group_list": counts,
        "x": normal_bf16(rng, (wl.M, wl.K)),
        "w": normal_bf16(rng, (wl.E, wl.K, wl.N), std=1.0 / np.sqrt(wl.K)),
    }
    if wl.backward:
        out["dy"] = normal_bf16(rng, (wl.M, wl.N))
    return out


def routing(rng: np.random.Generator, T: int, E: int, k: int, hot_bias: float = 0.0):
    """Router stand-in: N(0,1) logits (+hot_bias on one seeded expert), softmax,
    top-k (descending probability), weights renormalised to sum to one."""
    import torch
    logits = rng.standard_normal(size=(T, E), dtype=np.float32)
    hot = -1
    if hot_bias:
        hot = int(rng.integers(E))
        logits[:, hot] += np.float32(hot_bias)
    p = torch.softmax(torch.from_numpy(logits), dim=-1)
    vals, ids = torch.topk(p, k, dim=-1, largest=True, sorted=True)
    vals = vals / vals.sum(dim=-1, keepdim=True)
    return ids.to(torch.int32).numpy(), vals.to(torch.float32).numpy(), hot


def layer_inputs(wl: LayerWorkload, seed: Optional[int] = None, tokens: Optional[int] = None,
                 with_weights: bool = True) -> dict:
    """x[T,H], w1[E,H,2I], w2[E,I,H] (bf16 bits), topk_ids[T,k] int32, topk_w[T,k] float32,
    and dy[T,H] (bf16 bits) when the workload has a backward pass.

    ``tokens`` keeps only the first ``tokens`` rows of every per-token tensor
    (the draws are those of the full workload)."""
    rng = np.random.default_rng(wl.seed if seed is None else seed)
    ids, w, hot = routing(rng, wl.T, wl.E, wl.k, wl.hot_bias)
    x = normal_bf16(rng, (wl.T, wl.H))
    out = {"topk_ids": ids, "topk_w": w, "x": x, "hot_expert": hot}
    if wl.backward:
        out["dy"] = normal_bf16(rng, (wl.T, wl.H))
    if with_weights:
        # weights drawn from their own stream so token subsets never change them
        wrng = np.random.default_rng((wl.seed if seed is None else seed) + 1000)
        out["w1"] = normal_bf16(wrng, (wl.E, wl.H, 2 * wl.I), std=1.0 / np.sqrt(wl.H))
        out["w2"] = normal_bf16(wrng, (wl.E, wl.I, wl.H), std=1.0 / np.sqrt(wl.I))
    if tokens is not None:
        for key in ("topk_ids", "topk_w", "x", "dy"):
            if key in out:
                out[key] = np.ascontiguousarray(out[key][:tokens])
    return out


def fp8_codes(rng: np.random.Generator, shape, fmt: str = "e4m3", std: float = 16.0) -> np.ndarray:
    """N(0, std^2) draws cast to an fp8 type by torch's CPU conversion, as raw
    uint8 codes (fmt "e4m3" = float8_e4m3fn or "e5m2"); for "e2m1", codes
    uniform over all 16 (one per byte)."""
    if fmt == "e2m1":
        return rng.integers(0, 16, size=shape).astype(np.uint8)
    import torch
    dt = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}[fmt]
    a = rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std)
    return torch.from_numpy(a).to(dt).view(torch.uint8).numpy().copy()


def e8m0_codes(rng: np.random.Generator, shape, centre: int) -> np.ndarray:
    """Scale codes drawn uniformly from centre-1, centre, centre+1."""
    return rng.integers(centre - 1, centre + 2, size=shape).astype(np.uint8)


def mx_weight(rng: np.random.Generator, E: int, N: int, K: int, fmt: str = "e4m3"):
    """(codes [E, N, K], scales [E, N, K/32]) of an MX weight whose dequantised
    values have a standard deviation near 1/sqrt(K): fp8 codes ~ N(0, 16^2)
    cast by torch, or e2m1 codes uniform over all 16 (one code per byte here;
    see pack_fp4 for the CUDA layout)."""
    if fmt == "e2m1":
        centre = 127 - 1 - int(round(0.5 * np.log2(K)))
        codes = rng.integers(0, 16, size=(E, N, K)).astype(np.uint8)
        return codes, e8m0_codes(rng, (E, N, K // 32), centre)
    centre = 127 - 4 - int(round(0.5 * np.log2(K)))
    return fp8_codes(rng, (E, N, K), fmt), e8m0_codes(rng, (E, N, K // 32), centre)


def pack_fp4(codes: np.ndarray) -> np.ndarray:
    """4-bit codes [..., K] (one per byte) -> bytes [..., K/2], element 2i in the
    low nibble of byte i."""
    c = np.asarray(codes, dtype=np.uint8)
    return np.ascontiguousarray((c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)).astype(np.uint8)


def unpack_fp4(packed: np.ndarray) -> np.ndarray:
    """The inverse of pack_fp4: bytes [..., K/2] -> 4-bit codes [..., K]."""
    b = np.asarray(packed, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), np.uint8)
    out[..., 0::2] = b & 0xF
    out[..., 1::2] = b >> 4
    return out


def mx_layer_weights(wl: LayerWorkload, seed: Optional[int] = None, fmt: Optional[str] = None) -> dict:
    """w1_q [E, 2I, H], w1_s [E, 2I, H/32], w2_q [E, H, I], w2_s [E, H, I/32] (uint8)."""
    fmt = fmt or wl.w_mx or wl.mx or "e4m3"
    wrng = np.random.default_rng((wl.seed if seed is None else seed) + 2000)
    w1q, w1s = mx_weight(wrng, wl.E, 2 * wl.I, wl.H, fmt)
    w2q, w2s = mx_weight(wrng, wl.E, wl.H, wl.I, fmt)
    return {"w1_q": w1q, "w1_s": w1s, "w2_q": w2q, "w2_s": w2s}
