"""Seeded synthetic workloads for the sparsely-gated MoE FFN layer.

This module draws inputs and nothing else: shapes, seeds, random numbers and one
cast to the run dtype.  It holds none of the layer's arithmetic (no scoring,
selection, capacity or expert math), so both the CUDA path and the CPU oracle
can consume the same tensors without sharing any of the method.

Recipe (every workload): one torch.Generator per tensor, seeded with
``(20261202 + workload index) * 64 + tensor slot``, drawing fp32 values that are
cast once to the run dtype.  ``N(0, v)`` is read as mean 0, *variance* v, so
weights ~ N(0, 1/fan_in) have std 1/sqrt(fan_in).  Expert weights are drawn one
expert at a time (same generator, in expert order) to keep host/device peaks small.

The workloads follow the configurations the layer is measured on:
  * tiny top-2 softmax layer in fp32 (T=256, d=128, E=8, f=256, k=2);
  * Switch-style top-1 with capacity factor 1.25 (T=8192, d=1024, E=64, f=4096);
  * Mixtral-shaped top-2 (d=4096, E=8, f=14336) at T in {16, 256, 4096, 16384}
    with per-expert router logit offsets ~ N(0, 0.5);
  * DeepSeek-V3-shaped fine-grained layer (d=7168, 256 experts of f=2048, top-8
    sigmoid with a selection-only bias ~ U(-0.1, 0.1), one shared expert of f=2048);
  * Expert Choice under Zipf(1.1) skew (T=16384, d=2048, E=64, f=8192, cap=512).
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass

import torch

BASE_SEED = 20261202

# tensor slots (fixed order: x, W_r, offsets/bias, W1, W3, W2, shared)
_SLOT_X, _SLOT_WR, _SLOT_LOGIT_OFF, _SLOT_SEL_BIAS = 0, 1, 2, 3
_SLOT_W1, _SLOT_W3, _SLOT_W2 = 4, 5, 6
_SLOT_W1S, _SLOT_W3S, _SLOT_W2S = 7, 8, 9


@dataclass(frozen=True)
class Workload:
    name: str
    index: int            # seed offset of the workload
    T: int
    d: int
    E: int
    f: int
    k: int
    gate: str = "softmax"          # "softmax" | "sigmoid"
    mode: str = "tc"               # "tc" (token choice) | "ec" (expert choice)
    renorm: bool = True            # renormalise the selected k scores
    capacity_factor: float = 0.0   # <= 0: no capacity limit
    ec_capacity: int = 0           # expert choice: tokens per expert
    n_shared: int = 0
    f_shared: int = 0
    dtype: str = "bf16"            # "f32" | "bf16" | "fp8w" | "fp8up" (bf16 tensors; the library quantises)
    drop_policy: str = "token"     # capacity drop: "token" order or "affinity" (largest gate weights kept)
    logit_offsets: str = "none"    # "none" | "normal_var0.5" | "zipf1.1"
    sel_bias: str = "none"         # "none" | "uniform0.1"

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


WORKLOADS: dict[str, Workload] = {
    "tiny_top2_fp32": Workload("tiny_top2_fp32", 0, T=256, d=128, E=8, f=256, k=2,
                               renorm=True, dtype="f32"),
    "switch_top1_cap1.25": Workload("switch_top1_cap1.25", 1, T=8192, d=1024, E=64, f=4096,
                                    k=1, renorm=False, capacity_factor=1.25),
    "mixtral_T16": Workload("mixtral_T16", 2, T=16, d=4096, E=8, f=14336, k=2,
                            logit_offsets="normal_var0.5"),
    "mixtral_T256": Workload("mixtral_T256", 2, T=256, d=4096, E=8, f=14336, k=2,
                             logit_offsets="normal_var0.5"),
    "mixtral_T4096": Workload("mixtral_T4096", 2, T=4096, d=4096, E=8, f=14336, k=2,
                              logit_offsets="normal_var0.5"),
    "mixtral_T16384": Workload("mixtral_T16384", 2, T=16384, d=4096, E=8, f=14336, k=2,
                               logit_offsets="normal_var0.5"),
    "deepseek_v3": Workload("deepseek_v3", 3, T=4096, d=7168, E=256, f=2048, k=8,
                            gate="sigmoid", renorm=True, n_shared=1, f_shared=2048,
                            sel_bias="uniform0.1"),
    "expert_choice_zipf": Workload("expert_choice_zipf", 4, T=16384, d=2048, E=64, f=8192,
                                   k=0, mode="ec", ec_capacity=512, renorm=False,
                                   logit_offsets="zipf1.1"),
}


def _gen(w: Workload, slot: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((BASE_SEED + w.index) * 64 + slot)
    return g


def _normal(shape, std, g, device, dtype):
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _expert_stack(n, rows, cols, fan_in, slot, w, device, dtype):
    g = _gen(w, slot, device)
    out = torch.empty(n, rows, cols, device=device, dtype=dtype)
    std = 1.0 / math.sqrt(fan_in)
    for e in range(n):
        out[e].copy_(_normal((rows, cols), std, g, device, dtype))
    return out


def make_inputs(w: Workload, device="cpu", weights=True) -> dict:
    """Materialise the workload's tensors on ``device``.

    Returns x[T,d], W_r[d,E], logit_offset[E] (fp32 or None), sel_bias[E] (fp32 or
    None), W1/W3[E,d,f], W2[E,f,d] and, with shared experts, W1s/W3s[S,d,fs],
    W2s[S,fs,d].  The same seed always gives the same values on the same device.
    """
    dt = w.torch_dtype
    out = {}
    out["x"] = _normal((w.T, w.d), 1.0, _gen(w, _SLOT_X, device), device, dt)
    out["W_r"] = _normal((w.d, w.E), 1.0 / math.sqrt(w.d), _gen(w, _SLOT_WR, device), device, dt)

    g = _gen(w, _SLOT_LOGIT_OFF, device)
    if w.logit_offsets == "none":
        out["logit_offset"] = None
    elif w.logit_offsets == "normal_var0.5":
        out["logit_offset"] = torch.randn(w.E, generator=g, device=device) * math.sqrt(0.5)
    elif w.logit_offsets == "zipf1.1":
        # expert of popularity rank r gets offset -1.1 ln r: its unnormalised
        # affinity exp(u) is scaled by r^-1.1 (Zipf with s = 1.1); ranks are a
        # seeded permutation of 1..E
        rank = torch.randperm(w.E, generator=g, device=device).to(torch.float32) + 1.0
        out["logit_offset"] = -1.1 * torch.log(rank)
    else:
        raise ValueError(w.logit_offsets)

    g = _gen(w, _SLOT_SEL_BIAS, device)
    if w.sel_bias == "none":
        out["sel_bias"] = None
    elif w.sel_bias == "uniform0.1":
        out["sel_bias"] = torch.rand(w.E, generator=g, device=device) * 0.2 - 0.1
    else:
        raise ValueError(w.sel_bias)

    if weights:
        out["W1"] = _expert_stack(w.E, w.d, w.f, w.d, _SLOT_W1, w, device, dt)
        out["W3"] = _expert_stack(w.E, w.d, w.f, w.d, _SLOT_W3, w, device, dt)
        out["W2"] = _expert_stack(w.E, w.f, w.d, w.f, _SLOT_W2, w, device, dt)
        if w.n_shared > 0:
            out["W1s"] = _expert_stack(w.n_shared, w.d, w.f_shared, w.d, _SLOT_W1S, w, device, dt)
            out["W3s"] = _expert_stack(w.n_shared, w.d, w.f_shared, w.d, _SLOT_W3S, w, device, dt)
            out["W2s"] = _expert_stack(w.n_shared, w.f_shared, w.d, w.f_shared, _SLOT_W2S, w, device, dt)
    return out


def random_assignment(T: int, E: int, k: int, seed: int, skew: float = 0.0, device="cpu"):
    """A seeded routing table idx[T,k] of distinct experts per token.

    Used to drive the dispatch and combine stages with identical integer input on
    both sides.  ``skew`` > 0 draws experts with probability proportional to
    r^-skew (r = expert rank), so some experts overflow a capacity limit.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(BASE_SEED * 7 + seed)
    if skew > 0:
        p = (torch.arange(1, E + 1, dtype=torch.float64) ** (-skew))
    else:
        p = torch.ones(E, dtype=torch.float64)
    p = p / p.sum()
    idx = torch.multinomial(p.expand(T, E).contiguous(), k, replacement=False, generator=g)
    return idx.to(torch.int32).to(device)


def random_rows(n: int, d: int, seed: int, dtype=torch.bfloat16, device="cpu", std=1.0):
    g = torch.Generator(device="cpu")
    g.manual_seed(BASE_SEED * 11 + seed)
    return (torch.randn(n, d, generator=g) * std).to(dtype).to(device)


def random_weights(shape, seed: int, device="cpu"):
    """Seeded positive gate weights in [0.05, 1) for combine-stage tests."""
    g = torch.Generator(device="cpu")
    g.manual_seed(BASE_SEED * 13 + seed)
    return (torch.rand(*shape, generator=g) * 0.95 + 0.05).to(torch.float32).to(device)
