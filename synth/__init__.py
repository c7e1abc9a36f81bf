"""Seeded synthetic inputs for the ragged decode-attention path.

This module is the only code that both the CUDA path and the CPU oracle use.
It draws inputs and nothing else: per-head budgets B^, context lengths, token
scores, queries, keys and values.  None of the method's arithmetic (budget
scaling by alpha, top-k retention, paging, split maps, attention, page scores)
lives here.

Workloads (shapes and distributions) follow the five benchmark
configurations of the ragged paged decode-attention study:

  1. one Llama-3.1-8B-shaped layer, batch 1, N=4096, B ~ U[0.1, 1.0];
  2. Llama-3.1-8B shape, 32 layers, batch 16, N=32768, lognormal budgets
     (sigma 0.8) renormalised to mean 0.3 and clipped to (0, 1];
  3. Qwen3-4B-like skew stress, 36 layers, batch 4, N=100000, 10% of heads
     with B=1 and the rest U[0.03, 0.2];
  4. FlexiCache sparse decode, Llama-3.1-8B shape, batch 40, N=10000,
     per-page min/max keys, top-K in {64, 128} pages;
  5. Gemma-3-12B-like mixed lengths, 48 layers, 16 q / 8 KV heads, d=256,
     batch 32, N log-uniform in [4K, 64K], lognormal budgets (sigma 0.6)
     renormalised to mean 0.5, safety alpha=2.

Random draws: budgets and context lengths use numpy's PCG64 seeded with
``seed``; the tensors (scores, q, K, V) use torch's generator on the
requested device, seeded per (seed, layer, kind), so one layer can be
regenerated without the others.  Values drawn on the CPU and on a GPU differ
for the same seed, but every test hands the SAME tensor to both sides.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

__all__ = ["Workload", "CONFIGS", "workload", "budgets_hat", "contexts",
           "scores", "keys_values", "queries", "small"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    L: int            # layers
    batch: int        # requests in the decode batch
    H_q: int          # query heads
    H: int            # KV heads
    d: int            # head dim
    N: int            # context length (max when ``ctx_dist`` is log-uniform)
    P: int = 16       # tokens per page
    H_p: int = 4      # heads per page group
    alpha: float = 1.0
    cluster: bool = False
    budget_dist: str = "uniform"      # see budgets_hat()
    budget_args: tuple = (0.1, 1.0)
    ctx_dist: str = "fixed"           # "fixed" | "loguniform"
    ctx_min: int = 0
    n_cta: Optional[int] = None       # None = occupancy-derived
    topk_pages: tuple = ()            # config 4 only
    seed: int = 0

    @property
    def g(self) -> int:
        return self.H_q // self.H

    @property
    def G(self) -> int:
        return self.H // self.H_p

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    1: Workload("cfg1-llama8b-1layer-b1-n4096", L=1, batch=1, H_q=32, H=8, d=128,
                N=4096, P=16, H_p=4, budget_dist="uniform", budget_args=(0.1, 1.0),
                n_cta=148, seed=1001),
    2: Workload("cfg2-llama8b-32L-b16-n32768-rho0.3", L=32, batch=16, H_q=32, H=8,
                d=128, N=32768, P=16, H_p=4, budget_dist="lognormal",
                budget_args=(0.8, 0.3), seed=1002),
    3: Workload("cfg3-qwen3-4b-36L-b4-n100000-skew", L=36, batch=4, H_q=32, H=8,
                d=128, N=100000, P=16, H_p=4, budget_dist="skew",
                budget_args=(0.10, 0.03, 0.2), seed=1003),
    4: Workload("cfg4-flexicache-32L-b40-n10000", L=32, batch=40, H_q=32, H=8,
                d=128, N=10000, P=16, H_p=1, budget_dist="ones", budget_args=(),
                topk_pages=(64, 128), seed=1004),
    5: Workload("cfg5-gemma3-12b-48L-b32-n4k-64k", L=48, batch=32, H_q=16, H=8,
                d=256, N=65536, P=16, H_p=4, alpha=2.0, cluster=True,
                budget_dist="lognormal_alpha", budget_args=(0.6, 0.5),
                ctx_dist="loguniform", ctx_min=4096, seed=1005),
}


def workload(cfg: int, **overrides) -> Workload:
    return CONFIGS[cfg].replace(**overrides)


def small(**kw) -> Workload:
    """A small workload (a few hundred tokens per head) for fast parity runs."""
    base = Workload("small", L=2, batch=3, H_q=8, H=4, d=128, N=700, P=16, H_p=2,
                    budget_dist="uniform", budget_args=(0.05, 1.0),
                    ctx_dist="loguniform", ctx_min=1, seed=7)
    return base.replace(**kw)


def _rng(seed: int, *salt: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, *salt]))


def budgets_hat(w: Workload) -> np.ndarray:
    """Per-(layer, KV head) budgets B^ as float32 [L][H], before alpha.

    uniform:          B^ ~ U[lo, hi]
    lognormal:        X ~ LogN(0, sigma); B^ = clip(mean_target * X / mean(X), (0, 1])
    lognormal_alpha:  X ~ LogN(0, sigma); B^ = mean_target * X / mean(X)  (alpha applied later)
    skew:             a seeded fraction of all L*H heads get 1.0, the rest U[lo, hi]
    ones:             every head keeps its whole context
    """
    r = _rng(w.seed, 1)
    shape = (w.L, w.H)
    if w.budget_dist == "uniform":
        lo, hi = w.budget_args
        b = r.uniform(lo, hi, size=shape)
    elif w.budget_dist in ("lognormal", "lognormal_alpha"):
        sigma, mean_target = w.budget_args
        x = r.lognormal(0.0, sigma, size=shape)
        b = mean_target * x / x.mean()
        if w.budget_dist == "lognormal":
            b = np.minimum(b, 1.0)
    elif w.budget_dist == "skew":
        frac, lo, hi = w.budget_args
        b = r.uniform(lo, hi, size=shape).reshape(-1)
        n_full = int(round(frac * b.size))
        b[r.permutation(b.size)[:n_full]] = 1.0
        b = b.reshape(shape)
    elif w.budget_dist == "ones":
        b = np.ones(shape)
    else:
        raise ValueError(w.budget_dist)
    b = b.astype(np.float32)
    # a draw can never be exactly 0; keep B^ strictly positive in float32
    return np.maximum(b, np.float32(np.finfo(np.float32).tiny))


def contexts(w: Workload) -> np.ndarray:
    """Context length N_b of every request, int32 [batch]."""
    if w.ctx_dist == "fixed":
        return np.full(w.batch, w.N, dtype=np.int32)
    if w.ctx_dist == "loguniform":
        r = _rng(w.seed, 2)
        lo = max(w.ctx_min, 1)
        u = r.uniform(math.log(lo), math.log(w.N), size=w.batch)
        return np.clip(np.round(np.exp(u)), lo, w.N).astype(np.int32)
    raise ValueError(w.ctx_dist)


def _gen(w: Workload, layer: int, kind: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((w.seed * 1000003 + layer * 7919 + kind) % (2**63 - 1))
    return g


def scores(w: Workload, layer: int, device="cpu") -> torch.Tensor:
    """Token importance scores s_{l,h}: float32 N(0,1), [batch][H][N]."""
    return torch.randn((w.batch, w.H, w.N), generator=_gen(w, layer, 11, device),
                       device=device, dtype=torch.float32)


def keys_values(w: Workload, layer: int, device="cpu"):
    """Full-context K and V for one layer: bf16 N(0,1), [batch][H][N][d] each."""
    shape = (w.batch, w.H, w.N, w.d)
    k = torch.randn(shape, generator=_gen(w, layer, 12, device), device=device,
                    dtype=torch.float32 if device == "cpu" else torch.bfloat16)
    v = torch.randn(shape, generator=_gen(w, layer, 13, device), device=device,
                    dtype=torch.float32 if device == "cpu" else torch.bfloat16)
    return k.to(torch.bfloat16), v.to(torch.bfloat16)


def queries(w: Workload, layer: int, device="cpu", step: int = 0) -> torch.Tensor:
    """Decode-step queries: bf16 N(0,1), [batch][H_q][d]."""
    shape = (w.batch, w.H_q, w.d)
    q = torch.randn(shape, generator=_gen(w, layer, 14 + 17 * step, device), device=device,
                    dtype=torch.float32 if device == "cpu" else torch.bfloat16)
    return q.to(torch.bfloat16)
