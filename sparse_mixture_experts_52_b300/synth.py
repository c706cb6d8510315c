"""Seeded synthetic inputs for the MoE-layer workloads.

This module only draws numbers: it holds none of the layer's arithmetic, so
both the CUDA path and the CPU oracle can be fed from it.  Every tensor is
drawn in float32 from ``torch.Generator`` seeded per workload on the device
that will hold it, then (for bf16 workloads) rounded to bf16 once; a test hands
the very same values to both sides.

Recipe (per workload, in draw order): x ~ N(0, 1) [T, d]; W_g ~ N(0, 1/d)
[d, E]; per routed expert e = 0..E-1: W1_e ~ N(0, 1/d) [d_ff, d] ([2 d_ff, d]
for SwiGLU experts: gate rows, then up rows), then W2_e ~ N(0, 1/d_ff)
[d, d_ff]; then the shared experts in the same way; then
the optional biases and the DeepSeek-style selection bias ~ N(0, 0.01^2) [E].
Biases are zero unless ``nonzero_bias`` (then N(0, 0.1^2)).  The skewed decode
workload adds a fixed logit offset log(Zipf(s=1.2) over the experts), expert 0
most favoured.
"""

from __future__ import annotations

import math
from typing import Optional

import torch

# The five workloads: shapes, routing form and statistics as the layer's
# problem statement names them (T tokens, d_model, d_ff, E experts, top-k,
# capacity factor, routing variant).
WORKLOADS = {
    # tiny fp32 top-2 layer with (zero) biases; softmax -> top-2 -> renormalise
    "tiny_fp32_top2": dict(
        T=256, d_model=64, d_ff=256, E=8, k=2, n_shared=0, capacity_factor=0.0,
        min_capacity=0, route="softmax_topk", renorm=1, dtype="f32", has_bias=1,
        aux_alpha=0.01, aux_f="topk_count", seed=0, logit_bias=None,
        select_bias_std=0.0),
    # Switch-style top-1, capacity factor 1.25 (C = 80), argmax f_i
    "switch_top1_cap": dict(
        T=4096, d_model=768, d_ff=3072, E=64, k=1, n_shared=0,
        capacity_factor=1.25, min_capacity=0, route="softmax_topk", renorm=0,
        dtype="bf16", has_bias=0, aux_alpha=0.01, aux_f="argmax", seed=0,
        logit_bias=None, select_bias_std=0.0),
    # Mixtral-shaped: top-2 on logits then softmax over the 2
    "mixtral_top2": dict(
        T=8192, d_model=4096, d_ff=14336, E=8, k=2, n_shared=0,
        capacity_factor=0.0, min_capacity=0, route="topk_softmax", renorm=1,
        dtype="bf16", has_bias=0, aux_alpha=0.01, aux_f="topk_count", seed=0,
        logit_bias=None, select_bias_std=0.0),
    # DeepSeek-V3-shaped: 256 fine-grained experts + 1 shared, top-8 on
    # softmax + selection bias, weights from the unbiased scores renormalised
    "deepseek_v3_top8": dict(
        T=4096, d_model=7168, d_ff=2048, E=256, k=8, n_shared=1,
        capacity_factor=0.0, min_capacity=0, route="biased_softmax", renorm=1,
        dtype="bf16", has_bias=0, aux_alpha=0.01, aux_f="topk_count", seed=0,
        logit_bias=None, select_bias_std=0.01),
    # decode-shaped Mixtral layer, T = 64, Zipf(1.2) logit offset
    "decode_zipf_top2": dict(
        T=64, d_model=4096, d_ff=14336, E=8, k=2, n_shared=0,
        capacity_factor=0.0, min_capacity=0, route="topk_softmax", renorm=1,
        dtype="bf16", has_bias=0, aux_alpha=0.01, aux_f="topk_count", seed=0,
        logit_bias="zipf1.2", select_bias_std=0.0),
}

# The Mixtral shape with SwiGLU experts, the activation named for Mixtral's
# FFN (its W1 holds the gate and up projections: 2 x 14336 rows).
WORKLOADS["mixtral_swiglu_top2"] = dict(WORKLOADS["mixtral_top2"], act="swiglu")

# The Switch shape under Expert Choice routing: each of the 64 experts takes
# its C = floor(2.0 * 4096 / 64) = 128 highest-scoring tokens.
WORKLOADS["switch_expert_choice"] = dict(WORKLOADS["switch_top1_cap"], route="expert_choice",
                                         capacity_factor=2.0, aux_f="topk_count")

# MX FP8 experts (e4m3 weights and activations with 32-element power-of-two
# block scales): the weight-streaming Switch and decode shapes, where the
# weight bytes halve, and the compute-bound Mixtral shape.
for _name in ("switch_top1_cap", "decode_zipf_top2", "mixtral_top2"):
    WORKLOADS[_name + "_mxfp8"] = dict(WORKLOADS[_name], experts="mxfp8")

LAYER_KEYS = ("T", "d_model", "d_ff", "E", "k", "n_shared", "capacity_factor",
              "min_capacity", "route", "renorm", "dtype", "has_bias",
              "aux_alpha", "aux_f", "act", "y_f32", "experts")


def workload(name: str, **overrides) -> dict:
    """A copy of a named workload with some fields replaced."""
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    cfg["name"] = name
    return cfg


def zipf_log_offset(E: int, s: float) -> torch.Tensor:
    """log of the Zipf(s) probabilities over E items: log((e+1)^-s / H)."""
    w = torch.tensor([(e + 1.0) ** (-s) for e in range(E)], dtype=torch.float64)
    return torch.log(w / w.sum()).to(torch.float32)


def _draw(g: torch.Generator, shape, std: float, device, dtype) -> torch.Tensor:
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def make_inputs(cfg: dict, device="cpu", seed: Optional[int] = None,
                nonzero_bias: bool = False) -> dict:
    """Draw every input of one layer call on ``device``.

    Returns a dict of tensors: x, w_g, w1 [E,F1,d] (F1 = 2F for SwiGLU, else
    F), w2 [E,d,F], b1/b2 (or None),
    ws1/ws2/wsb1/wsb2 for shared experts (or None), logit_bias, select_bias
    (float32 [E] or None).
    """
    device = torch.device(device)
    seed = cfg.get("seed", 0) if seed is None else seed
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    dt = torch.float32 if cfg["dtype"] == "f32" else torch.bfloat16
    T, d, F, E, S = cfg["T"], cfg["d_model"], cfg["d_ff"], cfg["E"], cfg["n_shared"]
    F1 = 2 * F if cfg.get("act", "gelu") == "swiglu" else F   # rows of W1

    out = {}
    out["x"] = _draw(g, (T, d), 1.0, device, dt)
    out["w_g"] = _draw(g, (d, E), 1.0 / math.sqrt(d), device, dt)
    w1 = torch.empty((E, F1, d), device=device, dtype=dt)
    w2 = torch.empty((E, d, F), device=device, dtype=dt)
    for e in range(E):
        w1[e] = _draw(g, (F1, d), 1.0 / math.sqrt(d), device, dt)
        w2[e] = _draw(g, (d, F), 1.0 / math.sqrt(F), device, dt)
    out["w1"], out["w2"] = w1, w2
    if S > 0:
        ws1 = torch.empty((S, F1, d), device=device, dtype=dt)
        ws2 = torch.empty((S, d, F), device=device, dtype=dt)
        for s in range(S):
            ws1[s] = _draw(g, (F1, d), 1.0 / math.sqrt(d), device, dt)
            ws2[s] = _draw(g, (d, F), 1.0 / math.sqrt(F), device, dt)
        out["ws1"], out["ws2"] = ws1, ws2
    else:
        out["ws1"] = out["ws2"] = None

    out["b1"] = out["b2"] = out["wsb1"] = out["wsb2"] = None
    if cfg["has_bias"]:
        if nonzero_bias:
            out["b1"] = _draw(g, (E, F1), 0.1, device, dt)
            out["b2"] = _draw(g, (E, d), 0.1, device, dt)
            if S > 0:
                out["wsb1"] = _draw(g, (S, F1), 0.1, device, dt)
                out["wsb2"] = _draw(g, (S, d), 0.1, device, dt)
        else:
            out["b1"] = torch.zeros((E, F1), device=device, dtype=dt)
            out["b2"] = torch.zeros((E, d), device=device, dtype=dt)
            if S > 0:
                out["wsb1"] = torch.zeros((S, F1), device=device, dtype=dt)
                out["wsb2"] = torch.zeros((S, d), device=device, dtype=dt)

    sb = cfg.get("select_bias_std", 0.0)
    out["select_bias"] = (_draw(g, (E,), sb, device, torch.float32)
                          if cfg["route"] == "biased_softmax" and sb > 0 else None)
    lb = cfg.get("logit_bias")
    if lb is None:
        out["logit_bias"] = None
    elif isinstance(lb, str) and lb.startswith("zipf"):
        out["logit_bias"] = zipf_log_offset(E, float(lb[4:])).to(device)
    else:
        out["logit_bias"] = torch.as_tensor(lb, dtype=torch.float32, device=device)
    return out
