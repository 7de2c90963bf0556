"""Striped KV-cache layout and the KV write -- oracle side (test infrastructure).

Layout (a reading of "striped shard" in the PCP ring-cache PR, Design
section, and of its "strided KV cache write", Testing section): stripe width
one token, so token t of a sequence lives in shard ``t mod P`` at row
``t div P``.  The cache of all sequences is one array
``[B, NKV, P, S, HD]``; shard s of (b, kv head g) holds ``n_s(L)`` filled rows
``0 .. n_s(L)-1`` where n_s(L) = #{t < L : t mod P == s}.

The write is a pure bit copy of the chunk's valid tokens into their slots --
the same contract as the ``index_copy_`` scatter of the m-star
``ring_scatter`` op.  Values are handled as raw uint16 so that "bit-exact"
means exactly that.
"""
from __future__ import annotations

from typing import Sequence

import numpy as np


def shard_of_token(t, P: int):
    """(shard, row) of token position t under stripe width one."""
    return t % P, t // P


def shard_fill(L: int, P: int) -> np.ndarray:
    """n_s(L) for s = 0..P-1: how many of the first L tokens land in shard s."""
    if L == 0:
        return np.zeros(P, dtype=np.int64)
    t = np.arange(L)
    return np.bincount(t % P, minlength=P)[:P]


def _scatter(cache: np.ndarray, b: int, positions: np.ndarray, rows: np.ndarray, P: int, S: int):
    """cache[b, :, s(t), j(t), :] = rows[k] for t = positions[k]."""
    s, j = shard_of_token(positions, P)
    if positions.size and int(j.max()) >= S:
        raise IndexError(f"token {int(positions.max())} needs shard row {int(j.max())} >= S={S}")
    # rows: [n, NKV, HD];  cache[b][:, s, j, :] is [NKV, n, HD]
    cache[b][:, s, j, :] = np.swapaxes(rows, 0, 1)


def write_kv_ref(k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
                 cache_lens: Sequence[int], chunk_lens: Sequence[int], chunk: int,
                 v_f16: bool = False) -> None:
    """In-place KV write of one prefill step (operands as uint16 bit patterns).

    k_cache, v_cache: [B, NKV, P, S, HD];  k_new, v_new: [B*C, NKV, HD] in
    token order.  For each sequence b, the valid chunk tokens i < c_b go to
    token position t = L_b + i.  Pad rows (i >= c_b) and every other cache
    row are left untouched.  v_f16: the V cache holds binary16, and each bf16
    value of v_new is stored as ``bf16_to_f16_bits`` of it.
    """
    B, _, P, S, _ = k_cache.shape
    for b in range(B):
        L, c = int(cache_lens[b]), int(chunk_lens[b])
        if c == 0:
            continue
        pos = np.arange(L, L + c)
        src = slice(b * chunk, b * chunk + c)
        _scatter(k_cache, b, pos, k_new[src], P, S)
        _scatter(v_cache, b, pos, bf16_to_f16_bits(v_new[src]) if v_f16 else v_new[src], P, S)


def build_striped_cache(logical: Sequence[np.ndarray], num_kv_heads: int, P: int, S: int,
                        head_dim: int, fill, dtype=np.uint16) -> np.ndarray:
    """Place each sequence's logical cache [L_b, NKV, HD] into a fresh striped array.

    Rows that hold no token (holes, and the slots the coming chunk will take)
    keep ``fill``.
    """
    B = len(logical)
    cache = np.empty((B, num_kv_heads, P, S, head_dim), dtype=dtype)
    cache[...] = fill
    for b, rows in enumerate(logical):
        L = rows.shape[0]
        if L:
            _scatter(cache, b, np.arange(L), rows, P, S)
    return cache


def read_logical(cache: np.ndarray, b: int, L: int) -> np.ndarray:
    """Inverse of the layout: tokens 0..L-1 of sequence b as [L, NKV, HD]."""
    _, _, P, S, _ = cache.shape
    t = np.arange(L)
    s, j = shard_of_token(t, P)
    return np.swapaxes(cache[b][:, s, j, :], 0, 1)


def bf16_bits(x) -> np.ndarray:
    """Raw uint16 bit patterns of a torch bf16 tensor."""
    import torch
    return x.detach().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(u16: np.ndarray) -> np.ndarray:
    """Decode bf16 bit patterns (uint16) to float64 exactly (NaN patterns,
    signalling ones included, decode to NaN without a floating-point warning)."""
    with np.errstate(invalid="ignore"):
        return (np.asarray(u16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_to_f16_bits(u16: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> IEEE 754 binary16 bit patterns of the same values.

    The bf16 value (exact in float32) is rounded to the nearest binary16,
    ties to even, as IEEE 754 defines conversion to a narrower format:
    exact for normal values within binary16's range and, since a bf16 value
    has 8 significant bits, for subnormal results down to 2^-17; below that
    rounded to a multiple of 2^-24 (zero at or below 2^-25); +-inf beyond
    65504 + half an ulp.
    """
    f32 = (np.asarray(u16).astype(np.uint32) << 16).view(np.float32)
    with np.errstate(over="ignore"):
        return f32.astype(np.float16).view(np.uint16)


def f16_bits_to_f64(u16: np.ndarray) -> np.ndarray:
    """Decode binary16 bit patterns (uint16) to float64 exactly."""
    return np.asarray(u16, dtype=np.uint16).view(np.float16).astype(np.float64)
