"""Prefill with the KV-cache write fused into the same launch.

Two things must hold at once: the attention output meets the parity bar
against the fp64 oracle (the write never disturbs what the prefill reads),
and the caches afterwards equal the oracle's scatter of the chunk bit for bit
over the ENTIRE buffers (untouched rows keep their prior contents, guard
bands intact) -- the same contract as cpattn_write_kv.  Covered: ragged
multi-sequence cases at both head dims, empty caches and chunks, both
pairing forms, GQA group 1, and split-KV pieces (only the first piece of a
row block writes)."""
import numpy as np
import pytest
import torch

import oracle
import long_context_chunked_gb300 as cp
from gpu_helpers import DeviceCase, compare, to_f64
from helpers import make_case
from workloads import small

pytestmark = pytest.mark.gpu

CASES = [
    small("fw1", (0, 1000, 129, 3000), (300, 1, 256, 77), 320, nq=8, nkv=2, hd=128, shards=4,
          shard_capacity=1100, seed=71),
    small("fw2", (5000, 0, 1), (130, 0, 384), 384, nq=4, nkv=1, hd=256, shards=8,
          shard_capacity=800, seed=72),
    small("fw3", (700,), (200,), 256, nq=3, nkv=3, hd=128, shards=3, shard_capacity=400, seed=73),
    small("fw4", (127, 128, 129), (129, 128, 1), 129, nq=8, nkv=4, hd=256, shards=4,
          shard_capacity=200, seed=74),
]


def _run(w, split_tiles=None):
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    ws = None
    if split_tiles is not None:
        need, _ = ctx.splitkv_workspace(w.cache_lens, w.chunk_lens, split_tiles)
        ws = torch.empty(max(need // 4, 64), dtype=torch.float32, device="cuda")
        ctx.set_splitkv(ws, split_tiles)
    kc0, vc0 = dc.k_cache.bits().copy(), dc.v_cache.bits().copy()
    ctx.prefill_write_kv(w.cache_lens, w.chunk_lens, dc.q.t, dc.k_new.t, dc.v_new.t,
                         dc.k_cache.t, dc.v_cache.t, dc.out.t, dc.lse)
    assert ctx.sync_status() == 0, ctx.last_error()
    # The output: same bar as the plain prefill.
    ref, ref_lse = case.oracle_full()
    v = dc.valid_rows()
    compare(to_f64(dc.out.bits())[v], ref[v], f"{w.name} fused write")
    lse = dc.lse.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lse[v] - ref_lse[v])) < 2e-3, "LSE"
    # The caches: the oracle's scatter of the chunk onto the prior contents.
    kc_ref, vc_ref = kc0.copy(), vc0.copy()
    oracle.write_kv_ref(kc_ref, vc_ref, case.k_new_bits, case.v_new_bits, w.cache_lens,
                        w.chunk_lens, w.chunk)
    assert np.array_equal(dc.k_cache.bits(), kc_ref), "K cache differs from the oracle scatter"
    assert np.array_equal(dc.v_cache.bits(), vc_ref), "V cache differs from the oracle scatter"
    assert dc.guards_intact(), "write outside a buffer"


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_prefill_write_kv(w):
    _run(w)


@pytest.mark.parametrize("mode", ["none", "pingpong"])
def test_prefill_write_kv_pairing_modes(mode, monkeypatch):
    monkeypatch.setenv("CPATTN_PAIRING", mode)
    _run(CASES[0])


def test_prefill_write_kv_with_split_pieces():
    _run(CASES[0], split_tiles=3)
