"""The five seeded synthetic workloads of chunked-prefill GQA attention.

Each workload is one prefill step: every sequence b has ``cache_lens[b]``
tokens already in its KV cache and brings a new chunk of ``chunk_lens[b]``
tokens, padded to ``chunk`` rows.  The cache is stored as ``shards`` striped
shards of ``shard_capacity`` rows per (sequence, kv head).

Shapes follow the TPU PR "PCP: in-kernel ring cache phase, fused with the
current phase" (Performance section: NQ=32, NKV=2, HD=256, chunk 4k, 8 striped
shards) plus a small case and a ragged multi-sequence case.  Readings where the
pages leave a value open (shard count of the small and ragged cases, shard
capacity, the peaky-key recipe) are stated beside each field.

This module holds sizes and counting only; it contains none of the method's
arithmetic.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Tuple


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    cache_lens: Tuple[int, ...]      # L_b, tokens already cached per sequence
    chunk_lens: Tuple[int, ...]      # c_b <= chunk, valid rows of the new chunk
    chunk: int                       # C, padded rows per sequence
    num_q_heads: int                 # NQ
    num_kv_heads: int                # NKV
    head_dim: int                    # HD
    shards: int                      # P, stripe width one token
    shard_capacity: int              # S, rows per shard per (sequence, kv head)
    seed: int
    peaky_frac: float = 0.0          # fraction of token positions whose K is doubled
    description: str = ""

    @property
    def num_seqs(self) -> int:
        return len(self.cache_lens)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def tokens(self) -> int:
        """Rows of the token-order inputs Q / K_new / V_new (B * C)."""
        return self.num_seqs * self.chunk

    def valid_pairs_per_head(self) -> int:
        """Number of (query, key) pairs that are visible, per query head.

        Row i of sequence b sees the L_b cached keys and current keys 0..i.
        """
        return sum(c * L + c * (c + 1) // 2 for L, c in zip(self.cache_lens, self.chunk_lens))

    def attention_flops(self) -> int:
        """Algorithmic FLOPs: 2*HD for q.k plus 2*HD for p*v per visible pair."""
        return 4 * self.head_dim * self.num_q_heads * self.valid_pairs_per_head()

    def kv_write_bytes(self) -> int:
        """Algorithmic bytes of the KV write: K and V, read once and written once."""
        return 2 * 2 * sum(self.chunk_lens) * self.num_kv_heads * self.head_dim * 2

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _cap(cache_lens, chunk_lens, shards, pad=0) -> int:
    return max((L + c + shards - 1) // shards for L, c in zip(cache_lens, chunk_lens)) + pad


TINY = Workload(
    name="tiny",
    cache_lens=(512,), chunk_lens=(256,), chunk=256,
    num_q_heads=8, num_kv_heads=2, head_dim=128,
    # Shard count unstated for this case: P=2, one of the two counts the PR's
    # standalone check used.
    shards=2, shard_capacity=_cap((512,), (256,), 2),
    seed=0,
    description="1 sequence, cache 512 + chunk 256, NQ=8, NKV=2, HD=128, P=2",
)

CTX_8K = Workload(
    name="8k",
    cache_lens=(4096,), chunk_lens=(4096,), chunk=4096,
    num_q_heads=32, num_kv_heads=2, head_dim=256,
    shards=8, shard_capacity=1024,
    seed=1,
    description="cache 4096 + chunk 4096, NQ=32, NKV=2, HD=256, P=8 shards of 1024 rows",
)

CTX_32K = Workload(
    name="32k",
    cache_lens=(28672,), chunk_lens=(4096,), chunk=4096,
    num_q_heads=32, num_kv_heads=2, head_dim=256,
    shards=8, shard_capacity=4096,
    seed=2,
    # 1 % of the 32768 token positions (cache and chunk) get K doubled: a
    # peaky softmax.  Doubling is exact in bf16.
    peaky_frac=0.01,
    description="cache 28672 + chunk 4096, NQ=32, NKV=2, HD=256, P=8, K x2 on 1% of tokens",
)

CTX_128K = Workload(
    name="128k",
    cache_lens=(126976,), chunk_lens=(4096,), chunk=4096,
    num_q_heads=32, num_kv_heads=2, head_dim=256,
    # S = ceil((L + C) / P) + 16 = 16400, not a multiple of any power-of-two
    # tile height, so a flat walk over the shard rows puts tile edges across
    # shard boundaries.
    shards=8, shard_capacity=16400,
    seed=3,
    description="cache 126976 + chunk 4096, NQ=32, NKV=2, HD=256, P=8, S=16400",
)

VARLEN = Workload(
    name="varlen",
    cache_lens=(0, 777, 3000, 8192, 15000, 60001),
    chunk_lens=(4096, 4096, 1000, 4096, 37, 4096),
    chunk=4096,
    num_q_heads=32, num_kv_heads=4, head_dim=128,
    # P unstated: 8 gives unequal shard fill at L in {777, 3000, 15000, 60001}.
    # One S for the batch: ceil((60001 + 4096) / 8) = 8013.
    shards=8, shard_capacity=8013,
    seed=4,
    description="6 sequences, ragged cache and chunk lengths, NQ=32, NKV=4, HD=128, P=8, S=8013",
)

ALL = (TINY, CTX_8K, CTX_32K, CTX_128K, VARLEN)
BY_NAME = {w.name: w for w in ALL}


def small(name: str, cache_lens, chunk_lens, chunk, nq=4, nkv=2, hd=128, shards=2,
          shard_capacity=None, seed=100, peaky_frac=0.0) -> Workload:
    """A small ad-hoc workload (edge cases, oracle pins)."""
    cache_lens = tuple(int(x) for x in cache_lens)
    chunk_lens = tuple(int(x) for x in chunk_lens)
    if shard_capacity is None:
        shard_capacity = max(1, _cap(cache_lens, chunk_lens, shards))
    return Workload(name=name, cache_lens=cache_lens, chunk_lens=chunk_lens, chunk=chunk,
                    num_q_heads=nq, num_kv_heads=nkv, head_dim=hd, shards=shards,
                    shard_capacity=shard_capacity, seed=seed, peaky_frac=peaky_frac)


@dataclasses.dataclass(frozen=True)
class Request:
    """A whole chunked prefill of one batch of requests: step k brings
    ``steps[k][b]`` new tokens of sequence b (0..chunk), and its cache then
    holds every token of the earlier steps -- the PR's per-request cumulative
    prefill (Performance section), with the KV write of each chunk between
    the steps."""
    name: str
    steps: Tuple[Tuple[int, ...], ...]
    chunk: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    shards: int
    shard_capacity: int
    seed: int

    @property
    def num_seqs(self) -> int:
        return len(self.steps[0])

    def step(self, k: int) -> Workload:
        """Step k as a one-step workload (sizes only; its inputs come from
        ``generate_request``)."""
        cache = tuple(sum(s[b] for s in self.steps[:k]) for b in range(self.num_seqs))
        return Workload(name=f"{self.name}/{k}", cache_lens=cache, chunk_lens=self.steps[k],
                        chunk=self.chunk, num_q_heads=self.num_q_heads,
                        num_kv_heads=self.num_kv_heads, head_dim=self.head_dim,
                        shards=self.shards, shard_capacity=self.shard_capacity, seed=self.seed)


def request(name: str, steps, chunk, nq=4, nkv=2, hd=128, shards=3, seed=300,
            shard_capacity=None) -> Request:
    """A small cumulative request; the shard capacity defaults to the least
    that holds every sequence's whole request."""
    steps = tuple(tuple(int(x) for x in s) for s in steps)
    total = max(sum(s[b] for s in steps) for b in range(len(steps[0])))
    if shard_capacity is None:
        shard_capacity = max(1, -(-total // shards))
    return Request(name=name, steps=steps, chunk=chunk, num_q_heads=nq, num_kv_heads=nkv,
                   head_dim=hd, shards=shards, shard_capacity=shard_capacity, seed=seed)
