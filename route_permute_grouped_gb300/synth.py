"""Seeded synthetic inputs for the MoE layer.

This module only draws random numbers; it holds none of the layer's arithmetic.
Both the CUDA path's tests/benchmark and the fp64 checker are fed from it.

Every tensor has its own ``torch.Generator`` seeded with ``seed*1000 + id``; it
is drawn in fp32 and rounded to bf16 (round to nearest even) for bf16 tensors.
Large tensors are drawn on the device; the checker receives host copies of the
slices it needs.

Shapes mirror the models of "Scalable Training of Mixture-of-Experts Models
with Megatron Core" (DeepSeek-V3, Qwen3-235B; summary page "Modeling", captions
page Table 11) plus a Mixtral-8x7B-shaped layer and a tiny layer.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, asdict

import torch

# tensor ids inside one seed
X, ROUTER_W, W1, W3, W2, WS1, WS3, WS2, EXPERT_BIAS, LOGIT_PERM, DOUT, TOPK_KEYS = range(12)


@dataclass
class LayerShape:
    """One synthetic MoE layer: sizes, router options and value scales."""
    name: str
    T: int
    H: int
    E: int
    k: int
    F: int
    F_shared: int = 0
    score: str = "softmax"          # "softmax" or "sigmoid"
    n_groups: int = 1
    topk_groups: int = 1
    gate_scale: float = 1.0
    aux_coeff: float = 0.0
    expert_bias_range: float = 0.0  # expert_bias ~ U(-r, r) when r > 0
    skew: float = 0.0               # Zipf exponent of expert popularity (0 = balanced)
    w_std: float | None = None      # expert weight std (None: 1/sqrt(fan_in))
    inter_fp32: bool = False        # expert outputs / shared output kept in fp32
    out_fp32: bool = False          # layer output y (and dx) in fp32
    force_balanced: bool = False    # force-balanced routing (cyclic slot assignment)
    extra: dict = field(default_factory=dict)

    def as_dict(self):
        return asdict(self)


def shape(name: str, **over) -> LayerShape:
    """The named layer shapes."""
    base = {
        # tiny: fan-in scaled weights, the oracle finishes in milliseconds
        "tiny": dict(T=256, H=128, E=8, k=2, F=256),
        # Mixtral-8x7B-shaped: 8 experts, top-2, F=14336
        "mixtral": dict(T=16384, H=4096, E=8, k=2, F=14336, w_std=0.02, inter_fp32=True),
        # Qwen3-235B-shaped: 128 experts, top-8, F=1536
        "qwen3": dict(T=16384, H=4096, E=128, k=8, F=1536, w_std=0.02),
        # same shape, Zipf(1.2) expert popularity via a per-expert logit offset
        "qwen3_skew": dict(T=16384, H=4096, E=128, k=8, F=1536, w_std=0.02, skew=1.2),
        # DeepSeek-V3-shaped: 256 experts, top-8, sigmoid + selection bias,
        # 8 groups / top-4 groups, gate scale 2.5, one shared expert F=2048
        "dsv3": dict(T=8192, H=7168, E=256, k=8, F=2048, F_shared=2048, score="sigmoid",
                     n_groups=8, topk_groups=4, gate_scale=2.5, expert_bias_range=0.1,
                     w_std=0.02, inter_fp32=True),
        # training step of the Qwen3 shape (balanced / skewed), aux loss 1e-2
        "qwen3_train": dict(T=16384, H=4096, E=128, k=8, F=1536, w_std=0.02, aux_coeff=1e-2),
        "qwen3_skew_train": dict(T=16384, H=4096, E=128, k=8, F=1536, w_std=0.02,
                                 aux_coeff=1e-2, skew=1.2),
        # profiling case: the Qwen3 expert shape and rows per expert (1024)
        # with 32 experts, so the device holds about 2 GB
        "qwen3_e32": dict(T=4096, H=4096, E=32, k=8, F=1536, w_std=0.02),
        "qwen3_e32_train": dict(T=4096, H=4096, E=32, k=8, F=1536, w_std=0.02, aux_coeff=1e-2),
    }[name]
    base.update(over)
    return LayerShape(name=name, **base)


def _gen(seed: int, tid: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + tid)
    return g


def _normal_bf16(shp, std, seed, tid, device, chunk_rows=None):
    """N(0, std^2) drawn in fp32, rounded to bf16. Drawn in row chunks of the
    leading axis so the fp32 temporary stays small."""
    out = torch.empty(shp, dtype=torch.bfloat16, device=device)
    g = _gen(seed, tid, device)
    n0 = shp[0]
    step = chunk_rows or n0
    for s in range(0, n0, step):
        e = min(n0, s + step)
        out[s:e] = (torch.randn((e - s,) + tuple(shp[1:]), generator=g, device=device,
                                dtype=torch.float32) * std).to(torch.bfloat16)
    return out


def make_layer(ls: LayerShape, seed: int = 1234, device="cpu", training=None):
    """All inputs of one layer call as torch tensors on ``device``.

    x [T,H] bf16 ~ N(0,1); router_w [E,H] bf16 ~ N(0,1/H); W1, W3 [E,H,F] and
    W2 [E,F,H] bf16 ~ N(0, w_std^2) (or N(0, 1/fan_in)); shared Ws1, Ws3 [H,Fs],
    Ws2 [Fs,H]; expert_bias [E] fp32 ~ U(-r, r); logit_bias [E] fp32 =
    -skew * 1.25 * ln(pi(e) + 1) for a seeded permutation pi (expert popularity
    proportional to (pi(e)+1)^-skew, scaled so the Zipf head dominates; the
    1.25 is the temperature of the logit offset); dO [T,H] bf16 ~ N(0,1) when
    training."""
    T, H, E, F = ls.T, ls.H, ls.E, ls.F
    training = (ls.aux_coeff > 0) if training is None else training
    sd1 = ls.w_std if ls.w_std is not None else 1.0 / math.sqrt(H)
    sd2 = ls.w_std if ls.w_std is not None else 1.0 / math.sqrt(F)
    d = {
        "x": _normal_bf16((T, H), 1.0, seed, X, device, chunk_rows=4096),
        "router_w": _normal_bf16((E, H), 1.0 / math.sqrt(H), seed, ROUTER_W, device),
        "W1": _normal_bf16((E, H, F), sd1, seed, W1, device, chunk_rows=8),
        "W3": _normal_bf16((E, H, F), sd1, seed, W3, device, chunk_rows=8),
        "W2": _normal_bf16((E, F, H), sd2, seed, W2, device, chunk_rows=8),
        "expert_bias": None, "logit_bias": None, "Ws1": None, "Ws3": None, "Ws2": None,
        "dO": None,
    }
    if ls.F_shared:
        Fs = ls.F_shared
        sds1 = ls.w_std if ls.w_std is not None else 1.0 / math.sqrt(H)
        sds2 = ls.w_std if ls.w_std is not None else 1.0 / math.sqrt(Fs)
        d["Ws1"] = _normal_bf16((H, Fs), sds1, seed, WS1, device)
        d["Ws3"] = _normal_bf16((H, Fs), sds1, seed, WS3, device)
        d["Ws2"] = _normal_bf16((Fs, H), sds2, seed, WS2, device)
    if ls.expert_bias_range > 0:
        g = _gen(seed, EXPERT_BIAS, "cpu")
        r = ls.expert_bias_range
        d["expert_bias"] = ((torch.rand(E, generator=g) * 2 - 1) * r).to(device)
    if ls.skew > 0:
        g = _gen(seed, LOGIT_PERM, "cpu")
        pi = torch.randperm(E, generator=g).to(torch.float64)
        d["logit_bias"] = (-ls.skew * 1.25 * torch.log(pi + 1.0)).to(torch.float32).to(device)
    if training:
        d["dO"] = _normal_bf16((T, H), 1.0, seed, DOUT, device, chunk_rows=4096)
    return d


def synthetic_topk(T: int, E: int, k: int, seed: int = 1234, skew: float = 0.0,
                   device="cpu") -> torch.Tensor:
    """A routing decision drawn directly (for permute tests): k distinct experts
    per token, int32 [T,k]. Balanced: uniform random k-subsets. Skewed: experts
    drawn without replacement with weights proportional to (e+1)^-skew (Gumbel
    top-k of random keys)."""
    g = _gen(seed, TOPK_KEYS, "cpu")
    u = torch.rand((T, E), generator=g, dtype=torch.float64).clamp_(1e-12, 1 - 1e-12)
    keys = -torch.log(-torch.log(u))
    if skew > 0:
        keys = keys - skew * torch.log(torch.arange(1, E + 1, dtype=torch.float64))[None, :]
    idx = torch.argsort(keys, dim=1, descending=True, stable=True)[:, :k]
    return idx.to(torch.int32).to(device)
