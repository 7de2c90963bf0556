"""Seeded synthetic inputs for a :class:`workloads.configs.Workload`.

Everything is drawn on the CPU from one ``torch.Generator`` as N(0, 1) fp32
and rounded to bf16 (round to nearest even), in this order: Q, then per
sequence the logical cache K and V, then the new chunk's K and V, then the
peaky-key positions.  Arrays are in logical token order; neither the striped
cache layout nor any attention arithmetic lives here -- each consumer (the
oracle, the CUDA path) builds its own layout from these arrays.
"""
from __future__ import annotations

import dataclasses
from typing import List

import torch

from .configs import Request, Workload


@dataclasses.dataclass
class Inputs:
    q: torch.Tensor                 # [B*C, NQ, HD] bf16, token order, pad rows included
    k_new: torch.Tensor             # [B*C, NKV, HD] bf16
    v_new: torch.Tensor             # [B*C, NKV, HD] bf16
    k_cache: List[torch.Tensor]     # per sequence [L_b, NKV, HD] bf16, logical order
    v_cache: List[torch.Tensor]     # per sequence [L_b, NKV, HD] bf16
    peaky_positions: List[torch.Tensor]  # per sequence int64 positions in [0, L_b + c_b)


def _normal_bf16(gen: torch.Generator, *shape: int) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def generate(w: Workload, seed: int | None = None) -> Inputs:
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    T = w.tokens
    q = _normal_bf16(gen, T, w.num_q_heads, w.head_dim)
    k_cache, v_cache = [], []
    for L in w.cache_lens:
        k_cache.append(_normal_bf16(gen, L, w.num_kv_heads, w.head_dim))
        v_cache.append(_normal_bf16(gen, L, w.num_kv_heads, w.head_dim))
    k_new = _normal_bf16(gen, T, w.num_kv_heads, w.head_dim)
    v_new = _normal_bf16(gen, T, w.num_kv_heads, w.head_dim)

    peaky = []
    for b, (L, c) in enumerate(zip(w.cache_lens, w.chunk_lens)):
        n = L + c
        count = int(round(w.peaky_frac * n))
        if count:
            pos = torch.randperm(n, generator=gen)[:count].sort().values
        else:
            pos = torch.zeros(0, dtype=torch.int64)
        peaky.append(pos)
        if count:
            in_cache = pos[pos < L]
            in_chunk = pos[pos >= L] - L + b * w.chunk
            # x2 is exact in bf16 for these magnitudes.
            k_cache[b][in_cache] = k_cache[b][in_cache] * 2
            k_new[in_chunk] = k_new[in_chunk] * 2
    return Inputs(q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache,
                  peaky_positions=peaky)


@dataclasses.dataclass
class StepInputs:
    q: torch.Tensor       # [B*C, NQ, HD] bf16, token order, pad rows included
    k_new: torch.Tensor   # [B*C, NKV, HD] bf16
    v_new: torch.Tensor   # [B*C, NKV, HD] bf16


def generate_request(r: Request) -> List[StepInputs]:
    """Every step's chunk of a cumulative request, from one generator in step
    order: Q, then K_new, then V_new of each step (N(0, 1), bf16)."""
    gen = torch.Generator().manual_seed(r.seed)
    T = r.num_seqs * r.chunk
    out = []
    for _ in r.steps:
        q = _normal_bf16(gen, T, r.num_q_heads, r.head_dim)
        k = _normal_bf16(gen, T, r.num_kv_heads, r.head_dim)
        v = _normal_bf16(gen, T, r.num_kv_heads, r.head_dim)
        out.append(StepInputs(q=q, k_new=k, v_new=v))
    return out
