"""Shared test plumbing: oracle-side arrays for a workload (uses ``oracle``)."""
from __future__ import annotations

import dataclasses
import json
import os

import numpy as np

import oracle
from workloads import Workload, generate

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# bf16 bit patterns used to poison memory the kernels must not use.
POISON_BITS = np.uint16(0x4280)      # 64.0: large but finite
CANARY_BITS = np.uint16(0x7F7F)      # 3.39e38: finite, never a legal output


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@dataclasses.dataclass
class Case:
    w: Workload
    inputs: object
    q_bits: np.ndarray        # [T, NQ, HD] uint16
    k_new_bits: np.ndarray    # [T, NKV, HD]
    v_new_bits: np.ndarray
    k_cache_bits: np.ndarray  # [B, NKV, P, S, HD] striped, holes = POISON_BITS
    v_cache_bits: np.ndarray  # bf16, or binary16 when v_f16
    v_f16: bool = False

    def f64(self, name: str) -> np.ndarray:
        if name == "v_cache" and self.v_f16:
            return oracle.f16_bits_to_f64(self.v_cache_bits)
        return oracle.bits_to_f64(getattr(self, name + "_bits"))

    def oracle_full(self, threads: int = 1):
        w = self.w
        return oracle.attend_ref(self.f64("q"), self.f64("k_new"), self.f64("v_new"),
                                 self.f64("k_cache"), self.f64("v_cache"), w.cache_lens,
                                 w.chunk_lens, w.chunk, w.scale, threads=threads)

    def oracle_heads(self, heads):
        """The oracle's whole output for the listed q heads only: O [T,
        len(heads), HD] and LSE [T, len(heads)] (NaN pad rows), one q head at
        a time against its own kv head's keys, the heads run in parallel."""
        from concurrent.futures import ThreadPoolExecutor
        w = self.w
        G = w.num_q_heads // w.num_kv_heads
        vconv = oracle.f16_bits_to_f64 if self.v_f16 else oracle.bits_to_f64

        def one(h):
            g = oracle.kv_head_of(h, G)
            return oracle.attend_ref(
                oracle.bits_to_f64(self.q_bits[:, [h]]), oracle.bits_to_f64(self.k_new_bits[:, [g]]),
                oracle.bits_to_f64(self.v_new_bits[:, [g]]),
                oracle.bits_to_f64(self.k_cache_bits[:, [g]]), vconv(self.v_cache_bits[:, [g]]),
                w.cache_lens, w.chunk_lens, w.chunk, w.scale)

        with ThreadPoolExecutor(min(len(heads), os.cpu_count() or 1)) as ex:
            res = list(ex.map(one, heads))
        return (np.concatenate([o for o, _ in res], axis=1),
                np.concatenate([l for _, l in res], axis=1))

    def oracle_rows(self, samples):
        w = self.w
        vc = self.f64("v_cache") if self.v_f16 else self.v_cache_bits
        return oracle.attend_rows_ref(self.q_bits, self.k_new_bits, self.v_new_bits,
                                      self.k_cache_bits, vc, w.cache_lens,
                                      w.chunk_lens, w.chunk, w.scale, samples)


def make_case(w: Workload, hole_bits=POISON_BITS, v_f16: bool = False) -> Case:
    """v_f16: the V cache in binary16 (its bf16 values converted as the fp16
    cache write converts them; the oracle then reads V as stored)."""
    inp = generate(w)
    kc = oracle.build_striped_cache([oracle.bf16_bits(x) for x in inp.k_cache], w.num_kv_heads,
                                    w.shards, w.shard_capacity, w.head_dim, hole_bits)
    vc = oracle.build_striped_cache([oracle.bf16_bits(x) for x in inp.v_cache], w.num_kv_heads,
                                    w.shards, w.shard_capacity, w.head_dim, hole_bits)
    if v_f16:
        vc = oracle.bf16_to_f16_bits(vc)
    return Case(w=w, inputs=inp, q_bits=oracle.bf16_bits(inp.q),
                k_new_bits=oracle.bf16_bits(inp.k_new), v_new_bits=oracle.bf16_bits(inp.v_new),
                k_cache_bits=kc, v_cache_bits=vc, v_f16=v_f16)


def heads_per_kv_head(w: Workload, pairs: bool = True, seed: int = 99):
    """Seeded q heads to compare whole: for every kv head g, a pair of
    adjacent heads (2j, 2j + 1) of its group -- the two heads one CTA pair
    computes together -- or, pairs=False, one head (even for even g, odd for
    odd g, so both CTAs of a pair are covered across kv heads)."""
    rng = np.random.default_rng(seed)
    G = w.num_q_heads // w.num_kv_heads
    heads = []
    for g in range(w.num_kv_heads):
        j = int(rng.integers(max(G // 2, 1)))
        if G == 1:
            heads.append(g)
        elif pairs:
            heads += [g * G + 2 * j, g * G + 2 * j + 1]
        else:
            heads.append(g * G + 2 * j + (g & 1))
    return heads


def sample_rows(w: Workload, n: int, seed: int = 1234):
    """Seeded (token, q head) samples over valid rows: first/last rows of each
    sequence plus uniform draws."""
    rng = np.random.default_rng(seed)
    out = []
    for b, c in enumerate(w.chunk_lens):
        if c == 0:
            continue
        for i in sorted({0, c - 1, min(c - 1, 127), min(c - 1, 128)}):
            out.append((b * w.chunk + i, int(rng.integers(w.num_q_heads))))
    valid = [(b, c) for b, c in enumerate(w.chunk_lens) if c > 0]
    while len(out) < n:
        b, c = valid[int(rng.integers(len(valid)))]
        out.append((b * w.chunk + int(rng.integers(c)), int(rng.integers(w.num_q_heads))))
    return out
