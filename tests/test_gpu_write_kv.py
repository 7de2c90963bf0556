"""Strided KV-cache write on the GPU: bit-exact against the oracle's scatter
over the ENTIRE cache buffers (untouched rows keep their canaries), for all
five workloads and ragged edge cases."""
import numpy as np
import pytest
import torch

import oracle
import long_context_chunked_gb300 as cp
from gpu_helpers import Guarded
from workloads import ALL, small, generate

pytestmark = pytest.mark.gpu

HOLE = np.uint16(0x3F80)  # 1.0 in bf16: pre-existing cache contents


def _run(w):
    inp = generate(w)
    kn = oracle.bf16_bits(inp.k_new)
    vn = oracle.bf16_bits(inp.v_new)
    shape = (w.num_seqs, w.num_kv_heads, w.shards, w.shard_capacity, w.head_dim)
    rng = np.random.default_rng(w.seed)
    kc0 = rng.integers(0, 0x7F00, size=shape, dtype=np.uint16)   # arbitrary prior contents
    vc0 = rng.integers(0, 0x7F00, size=shape, dtype=np.uint16)
    ctx = cp.Context.for_workload(w)
    d_kn, d_vn = Guarded(kn.shape, kn), Guarded(vn.shape, vn)
    d_kc, d_vc = Guarded(shape, kc0), Guarded(shape, vc0)
    ctx.write_kv(w.cache_lens, w.chunk_lens, d_kn.t, d_vn.t, d_kc.t, d_vc.t)
    assert ctx.sync_status() == 0, ctx.last_error()
    kc_ref, vc_ref = kc0.copy(), vc0.copy()
    oracle.write_kv_ref(kc_ref, vc_ref, kn, vn, w.cache_lens, w.chunk_lens, w.chunk)
    assert np.array_equal(d_kc.bits(), kc_ref), "K cache differs from the oracle scatter"
    assert np.array_equal(d_vc.bits(), vc_ref), "V cache differs from the oracle scatter"
    for g in (d_kn, d_vn, d_kc, d_vc):
        assert g.guards_intact(), "write outside the buffers"


@pytest.mark.parametrize("w", ALL, ids=[w.name for w in ALL])
def test_write_kv_bit_exact(w):
    _run(w)


EDGE = [
    small("e1", (0,), (1,), 1, nq=2, nkv=1, hd=128, shards=1),
    small("e2", (3, 0, 9), (5, 0, 7), 8, nq=4, nkv=2, hd=256, shards=3),
    small("e3", (127, 128, 129), (129, 128, 1), 129, nq=8, nkv=4, hd=128, shards=4,
          shard_capacity=200),
    small("e4", (1000,), (333,), 400, nq=4, nkv=2, hd=256, shards=8, shard_capacity=167),
]


@pytest.mark.parametrize("w", EDGE, ids=[w.name for w in EDGE])
def test_write_kv_edges(w):
    _run(w)
