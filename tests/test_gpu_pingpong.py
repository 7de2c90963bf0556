"""The two-query-tile prefill kernel (CPATTN_PAIRING=pingpong, HD = 128)
against the fp64 oracle.

One CTA holds the query tiles of two adjacent q heads of one kv head and
alternates their products on the tensor core while the other head's softmax
runs; every K/V tile in shared memory serves both.  Covered: ragged
multi-sequence cases, GQA groups 2, 4 and 8, more head pairs than CTAs (each
CTA runs several rounds, so the query-tile and O barriers turn over), both P
precisions and both V cache formats, split-KV pieces, the fused KV write, the
full-size mixed-length workload on sampled rows, repeatability, and a bounded
wait that expires."""
import numpy as np
import pytest
import torch

import long_context_chunked_gb300 as cp
from gpu_helpers import DeviceCase, compare, to_f64
from helpers import make_case, sample_rows
from workloads import VARLEN, small

pytestmark = pytest.mark.gpu

CASES = [
    small("ppA", (0, 1000, 129, 3000), (300, 1, 256, 77), 320, nq=8, nkv=2, hd=128, shards=4,
          shard_capacity=1100, seed=201),
    small("ppB", (5000,), (640,), 640, nq=4, nkv=2, hd=128, shards=8, seed=202),
    small("ppC", (777, 60), (1000, 37), 1024, nq=16, nkv=2, hd=128, shards=8, seed=203,
          peaky_frac=0.02),
    # 32 q heads x 21 row blocks: 336 head pairs, up to three rounds per CTA
    small("ppD", (1500, 129), (2048, 640), 2048, nq=32, nkv=4, hd=128, shards=8, seed=204),
]


@pytest.fixture(autouse=True)
def _pingpong(monkeypatch):
    monkeypatch.setenv("CPATTN_PAIRING", "pingpong")


def _check(w, dc, case, fast_p=False, tag=""):
    ref, ref_lse = case.oracle_full()
    v = dc.valid_rows()
    out = to_f64(dc.out.bits())
    if fast_p:
        compare(out[v], ref[v], f"{w.name}{tag} fast_p", max_abs_bar=2e-2, rel_bar=3.5e-3)
    else:
        compare(out[v], ref[v], f"{w.name}{tag}")
    lse = dc.lse.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lse[v] - ref_lse[v])) < 2e-3, "LSE"
    pad = ~v
    if pad.any():
        assert np.all(dc.out.bits()[pad] == np.uint16(0x7F7F)), "pad rows written"
    assert dc.guards_intact(), "write outside a buffer"


@pytest.mark.parametrize("v_f16", [False, True], ids=["bf16_v", "f16_v"])
@pytest.mark.parametrize("fast_p", [False, True], ids=["accurate", "fast_p"])
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_pingpong_parity(w, fast_p, v_f16):
    case = make_case(w, v_f16=v_f16)
    dc = DeviceCase(case)
    dc.prefill(cp.Context.for_workload(w, fast_p=fast_p, v_cache_f16=v_f16))
    _check(w, dc, case, fast_p)


def test_pingpong_repeatable():
    """Identical bits on every launch: a race between the two query tiles'
    barriers or TMEM regions would show as run-to-run differences."""
    w = CASES[2]
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    dc.prefill(ctx)
    first = dc.out.bits().copy()
    for _ in range(3):
        dc.prefill(ctx)
        assert np.array_equal(first, dc.out.bits())


@pytest.mark.parametrize("t", [1, 3])
def test_pingpong_split_pieces(t):
    w = CASES[0]
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    need, blocks = ctx.splitkv_workspace(w.cache_lens, w.chunk_lens, t)
    assert need > 0 and blocks > sum(-(-c // 128) for c in w.chunk_lens)
    ws = torch.empty(max(need // 4, 64), dtype=torch.float32, device="cuda")
    ctx.set_splitkv(ws, t)
    dc.prefill(ctx)
    _check(w, dc, case, tag=f" split {t}")


@pytest.mark.parametrize("v_f16", [False, True], ids=["bf16_v", "f16_v"])
def test_pingpong_fused_write_kv(v_f16):
    import oracle
    w = CASES[0]
    case = make_case(w, v_f16=v_f16)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w, v_cache_f16=v_f16)
    kc0, vc0 = dc.k_cache.bits().copy(), dc.v_cache.bits().copy()
    ctx.prefill_write_kv(w.cache_lens, w.chunk_lens, dc.q.t, dc.k_new.t, dc.v_new.t,
                         dc.k_cache.t, dc.v_cache.t, dc.out.t, dc.lse)
    assert ctx.sync_status() == 0, ctx.last_error()
    _check(w, dc, case, tag=" fused write")
    kc_ref, vc_ref = kc0.copy(), vc0.copy()
    oracle.write_kv_ref(kc_ref, vc_ref, case.k_new_bits, case.v_new_bits, w.cache_lens,
                        w.chunk_lens, w.chunk, v_f16=v_f16)
    assert np.array_equal(dc.k_cache.bits(), kc_ref), "K cache differs from the oracle scatter"
    assert np.array_equal(dc.v_cache.bits(), vc_ref), "V cache differs from the oracle scatter"


def test_pingpong_full_size_sampled():
    """The mixed-length workload (6 sequences, HD = 128) at full size, in the
    launch configuration the benchmark times with this mode, on sampled rows."""
    w = VARLEN
    case = make_case(w, v_f16=True)
    dc = DeviceCase(case)
    dc.prefill(cp.Context.for_workload(w, v_cache_f16=True))
    samples = sample_rows(w, 48, seed=w.seed)
    ref, ref_lse = case.oracle_rows(samples)
    out = to_f64(dc.out.bits())
    got = np.stack([out[t, h] for t, h in samples])
    compare(got, ref, f"{w.name} pingpong")
    lse = dc.lse.cpu().numpy()
    assert np.max(np.abs(np.array([lse[t, h] for t, h in samples]) - ref_lse)) < 2e-3
    v = dc.valid_rows()
    assert np.all(np.isfinite(out[v])), "non-finite output"
    assert dc.guards_intact()


def test_pingpong_bounded_wait_reports_timeout():
    """One skipped P-ready arrival: the CTA's roles give up after the short
    limit, the host reads E_TIMEOUT, and the context computes correctly
    afterwards."""
    w = small("ppfail", (300,), (256,), 256, nq=4, nkv=2, hd=128, shards=2, seed=205)
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    ctx.set_fault_injection(1, timeout_ms=50)
    ctx.prefill(w.cache_lens, w.chunk_lens, dc.q.t, dc.k_new.t, dc.v_new.t, dc.k_cache.t,
                dc.v_cache.t, dc.out.t)
    assert ctx.sync_status() == cp.E_TIMEOUT
    assert ctx.sync_status() == cp.OK
    ctx.set_fault_injection(0, 0)
    dc.prefill(ctx)
    _check(w, dc, case, tag=" after timeout")
