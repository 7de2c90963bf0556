"""GQA packing on the GPU against the fp64 oracle.

When every chunk of a launch has at most 64 tokens and the group size G is a
power of two, a unit's 128 rows are (token, q head) pairs of one kv head: a
decode step fills 128 / G tokens x G heads instead of 1 row of 128.  Causal
visibility is then per row's own token, and outputs scatter back to (token,
head).  Checked at G = 2..16, both head dims, chunks of 1..64 tokens over
empty and long caches, with and without split-KV, with the fused KV write,
and against the unpacked kernel on the same inputs."""
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
    small("pk16", (20000, 0, 9000, 130), (1, 5, 37, 64), 64, nq=32, nkv=2, hd=256, shards=8,
          seed=81),
    small("pk8", (3000, 129), (8, 64), 64, nq=16, nkv=2, hd=128, shards=4, seed=82),
    small("pk4", (1000, 5000), (3, 17), 32, nq=8, nkv=2, hd=256, shards=8, seed=83),
    small("pk2", (0, 777), (64, 1), 64, nq=4, nkv=2, hd=128, shards=2, seed=84),
]


def _check(w, dc, case):
    ref, ref_lse = case.oracle_full()
    v = dc.valid_rows()
    out = to_f64(dc.out.bits())
    compare(out[v], ref[v], w.name)
    lse = dc.lse.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lse[v] - ref_lse[v])) < 2e-3, "LSE"
    pad = ~v
    if pad.any():
        assert np.all(dc.out.bits()[pad] == np.uint16(0x7F7F)), "pad rows written"
    assert dc.guards_intact(), "write outside a buffer"
    return out


def _packed_blocks(w):
    tb = 128 // (w.num_q_heads // w.num_kv_heads)
    return sum(-(-c // tb) for c in w.chunk_lens)


@pytest.mark.parametrize("split", [None, 0, 3], ids=["fused", "auto_split", "split3"])
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_packed_parity(w, split):
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    # The launch is packed: its row blocks are token blocks of 128 / G tokens.
    _, blocks = ctx.splitkv_workspace(w.cache_lens, w.chunk_lens, 1 << 20)
    assert blocks == _packed_blocks(w)
    if split is not None:
        need, _ = ctx.splitkv_workspace(w.cache_lens, w.chunk_lens, split)
        ws = torch.empty(max(need // 4, 64), dtype=torch.float32, device="cuda")
        ctx.set_splitkv(ws, split)
    dc.prefill(ctx)
    _check(w, dc, case)


def test_packed_and_unpacked_agree(monkeypatch):
    w = CASES[0]
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    dc.prefill(ctx)
    packed = _check(w, dc, case)
    monkeypatch.setenv("CPATTN_GQA_PACKING", "off")
    ctx2 = cp.Context.for_workload(w)
    _, blocks = ctx2.splitkv_workspace(w.cache_lens, w.chunk_lens, 1 << 20)
    assert blocks == sum(-(-c // 128) for c in w.chunk_lens)  # not packed
    dc2 = DeviceCase(case)
    dc2.prefill(ctx2)
    unpacked = _check(w, dc2, case)
    v = dc.valid_rows()
    d = np.abs(packed[v] - unpacked[v])
    assert float(d.max()) <= 2e-2 and float(np.sqrt((d * d).mean())) < 2e-3


@pytest.mark.parametrize("w", CASES[:2], ids=[w.name for w in CASES[:2]])
def test_packed_fused_kv_write(w):
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    kc0, vc0 = dc.k_cache.bits().copy(), dc.v_cache.bits().copy()
    ctx.prefill_write_kv(w.cache_lens, w.chunk_lens, dc.q.t, dc.k_new.t, dc.v_new.t,
                         dc.k_cache.t, dc.v_cache.t, dc.out.t, dc.lse)
    assert ctx.sync_status() == 0, ctx.last_error()
    _check(w, dc, case)
    kc_ref, vc_ref = kc0.copy(), vc0.copy()
    oracle.write_kv_ref(kc_ref, vc_ref, case.k_new_bits, case.v_new_bits, w.cache_lens,
                        w.chunk_lens, w.chunk)
    assert np.array_equal(dc.k_cache.bits(), kc_ref), "K cache differs from the oracle scatter"
    assert np.array_equal(dc.v_cache.bits(), vc_ref), "V cache differs from the oracle scatter"
