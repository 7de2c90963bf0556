"""fp16 V cache on the GPU against the fp64 oracle.

With cpattn_config.v_cache_f16 the KV write stores each V value converted to
binary16, and prefill takes P in fp16 for cache tiles: one P.V product per 16
keys instead of the bf16 hi + lo pair.  With a V staging buffer registered
("staged"), the chunk's own V is converted to fp16 too and its tiles take
fp16 P as well.  The oracle reads the cache's V as stored and the chunk's V
as the original bf16 values (the conversion is exact for them down to
2^-17).  Bar as everywhere: max |diff| <= 1e-2 and relative RMS <= 2e-3.
Checked over both head dims, paired / unpaired / two-tile CTAs, GQA packing,
split-KV, the fused KV write, the two-launch variant, fast_p on and off,
staged and not, the full-size workloads, the bit-exact fp16 cache write and
the range errors of the write and of the staging."""
import numpy as np
import pytest
import torch

import oracle
import long_context_chunked_gb300 as cp
from gpu_helpers import DeviceCase, compare, to_f64
from helpers import heads_per_kv_head, make_case, sample_rows
from workloads import CTX_8K, CTX_32K, CTX_128K, VARLEN, small

pytestmark = pytest.mark.gpu


def _ctx(w, staged, **kw):
    """Context with an fp16 V cache, and (staged) a V staging buffer for
    the workload's batch."""
    ctx = cp.Context.for_workload(w, v_cache_f16=True, **kw)
    if staged:
        n = ctx.v_staging_bytes(w.num_seqs)
        ctx._v_stage = torch.empty(n // 2, dtype=torch.float16, device="cuda")
        ctx.set_v_staging(ctx._v_stage)
    return ctx

CASES = [
    small("f16a", (0, 1000, 129, 3000), (300, 1, 256, 77), 320, nq=8, nkv=2, hd=128, shards=4,
          shard_capacity=800, seed=141),
    small("f16b", (5000, 1), (130, 384), 384, nq=4, nkv=1, hd=256, shards=8, seed=142),
    small("f16c", (2000,), (200,), 256, nq=3, nkv=3, hd=128, shards=3, seed=143),  # unpaired
    small("f16d", (20000, 0, 9000), (1, 5, 64), 64, nq=32, nkv=2, hd=256, shards=8,
          seed=144),  # GQA-packed
]


def _check(w, dc, case, fast_p=False):
    ref, ref_lse = case.oracle_full()
    v = dc.valid_rows()
    out = to_f64(dc.out.bits())
    if fast_p:
        # Current-chunk tiles then take P rounded once to bf16, whose error
        # floor (~2.2e-3 relative RMS) is above the bar: fast_p's own bound.
        res = compare(out[v], ref[v], f"{w.name} fast_p", max_abs_bar=2e-2, rel_bar=3.5e-3)
    else:
        res = compare(out[v], ref[v], w.name)
    lse = dc.lse.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lse[v] - ref_lse[v])) < 2e-3, "LSE"
    pad = ~v
    if pad.any():
        assert np.all(dc.out.bits()[pad] == np.uint16(0x7F7F)), "pad rows written"
    assert dc.guards_intact(), "write outside a buffer"
    return res


@pytest.mark.parametrize("staged", [False, True], ids=["bf16cur", "staged"])
@pytest.mark.parametrize("fast_p", [False, True], ids=["accurate", "fast_p"])
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_parity(w, fast_p, staged):
    case = make_case(w, v_f16=True)
    dc = DeviceCase(case)
    ctx = _ctx(w, staged, fast_p=fast_p)
    dc.prefill(ctx)
    _check(w, dc, case, fast_p)


@pytest.mark.parametrize("staged", [False, True], ids=["bf16cur", "staged"])
@pytest.mark.parametrize("mode", ["mma2", "none", "pingpong"])
def test_pairing_modes(mode, staged, monkeypatch):
    monkeypatch.setenv("CPATTN_PAIRING", mode)
    w = CASES[0]
    case = make_case(w, v_f16=True)
    dc = DeviceCase(case)
    dc.prefill(_ctx(w, staged))
    _check(w, dc, case)


@pytest.mark.parametrize("staged", [False, True], ids=["bf16cur", "staged"])
@pytest.mark.parametrize("t", [1, 3])
def test_split_kv(t, staged):
    w = CASES[1]
    case = make_case(w, v_f16=True)
    dc = DeviceCase(case)
    ctx = _ctx(w, staged)
    need, _ = ctx.splitkv_workspace(w.cache_lens, w.chunk_lens, t)
    ws = torch.empty(max(need // 4, 64), dtype=torch.float32, device="cuda")
    ctx.set_splitkv(ws, t)
    dc.prefill(ctx)
    _check(w, dc, case)


def test_more_accurate_than_single_bf16_p():
    """fp16 P on cache tiles carries 11 significand bits: on a cache-heavy
    case its error stays at the accurate mode's level, below the
    single-bf16-P (fast_p, bf16 cache) error."""
    w = small("f16acc", (6000,), (256,), 256, nq=4, nkv=2, hd=128, shards=8, seed=145)
    errs = {}
    for name, f16, fast in (("f16", True, False), ("bf16_fast", False, True)):
        case = make_case(w, v_f16=f16)
        dc = DeviceCase(case)
        dc.prefill(cp.Context.for_workload(w, fast_p=fast, v_cache_f16=f16))
        ref, _ = case.oracle_full()
        v = dc.valid_rows()
        errs[name] = compare(to_f64(dc.out.bits())[v], ref[v], name, rel_bar=3e-3)[1]
    assert errs["f16"] < 0.9 * errs["bf16_fast"], errs


def test_write_kv_bit_exact():
    w = CASES[0]
    case = make_case(w, v_f16=True)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w, v_cache_f16=True)
    kc_ref, vc_ref = case.k_cache_bits.copy(), case.v_cache_bits.copy()
    oracle.write_kv_ref(kc_ref, vc_ref, case.k_new_bits, case.v_new_bits, w.cache_lens,
                        w.chunk_lens, w.chunk, v_f16=True)
    ctx.write_kv(w.cache_lens, w.chunk_lens, dc.k_new.t, dc.v_new.t, dc.k_cache.t, dc.v_cache.t)
    assert ctx.sync_status() == cp.OK, ctx.last_error()
    assert np.array_equal(dc.k_cache.bits(), kc_ref), "K cache differs from the oracle scatter"
    assert np.array_equal(dc.v_cache.bits(), vc_ref), "V cache differs from the oracle scatter"
    assert dc.guards_intact()


@pytest.mark.parametrize("staged", [False, True], ids=["bf16cur", "staged"])
def test_fused_write_kv(staged):
    w = CASES[0]
    case = make_case(w, v_f16=True)
    dc = DeviceCase(case)
    ctx = _ctx(w, staged)
    kc_ref, vc_ref = case.k_cache_bits.copy(), case.v_cache_bits.copy()
    oracle.write_kv_ref(kc_ref, vc_ref, case.k_new_bits, case.v_new_bits, w.cache_lens,
                        w.chunk_lens, w.chunk, v_f16=True)
    ctx.prefill_write_kv(w.cache_lens, w.chunk_lens, dc.q.t, dc.k_new.t, dc.v_new.t,
                         dc.k_cache.t, dc.v_cache.t, dc.out.t, dc.lse)
    assert ctx.sync_status() == cp.OK, ctx.last_error()
    _check(w, dc, case)
    assert np.array_equal(dc.k_cache.bits(), kc_ref), "K cache differs from the oracle scatter"
    assert np.array_equal(dc.v_cache.bits(), vc_ref), "V cache differs from the oracle scatter"


def test_range_error_reported():
    """A V value beyond binary16's range (1e5) written to an fp16 cache makes
    the next status read CPATTN_E_RANGE; the status word is then clear."""
    w = small("f16rng", (100,), (40,), 64, nq=2, nkv=1, hd=128, shards=2, seed=146)
    case = make_case(w, v_f16=True)
    case.v_new_bits[7, 0, 5] = np.uint16(0x47C3)  # bf16 99840
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w, v_cache_f16=True)
    ctx.write_kv(w.cache_lens, w.chunk_lens, dc.k_new.t, dc.v_new.t, dc.k_cache.t, dc.v_cache.t)
    assert ctx.sync_status() == cp.E_RANGE
    assert ctx.sync_status() == cp.OK
    # The same write into a bf16 cache is a plain copy: no error.
    ctx16 = cp.Context.for_workload(w)
    dc2 = DeviceCase(make_case(w))
    ctx16.write_kv(w.cache_lens, w.chunk_lens, dc.k_new.t, dc.v_new.t, dc2.k_cache.t,
                   dc2.v_cache.t)
    assert ctx16.sync_status() == cp.OK


def test_staged_two_launch():
    """The two-launch variant stages V as the fused launch does."""
    w = CASES[0]
    case = make_case(w, v_f16=True)
    dc = DeviceCase(case)
    ctx = _ctx(w, True)
    ws = torch.empty(ctx.two_launch_workspace(w.num_seqs), dtype=torch.uint8, device="cuda")
    ctx.prefill_two_launch(w.cache_lens, w.chunk_lens, dc.q.t, dc.k_new.t, dc.v_new.t,
                           dc.k_cache.t, dc.v_cache.t, dc.out.t, ws, dc.lse)
    assert ctx.sync_status() == cp.OK, ctx.last_error()
    _check(w, dc, case)


def test_staged_range():
    """Staging converts the chunk's valid V rows as the fp16 cache write
    does: a value beyond binary16's range in a valid row makes the next
    status read CPATTN_E_RANGE.  Pad rows are staged as zeros: a huge finite
    value there is no error and cannot reach a valid row as NaN (0 x inf)."""
    w = small("f16srng", (300, 50), (40, 70), 128, nq=4, nkv=2, hd=128, shards=2, seed=147)
    case = make_case(w, v_f16=True)
    case.v_new_bits[100, 1, 9] = np.uint16(0x7F00)  # sequence 0, pad row 100: bf16 1.7e38
    case.v_new_bits[128 + 90, 0, 3] = np.uint16(0x7F00)  # sequence 1, pad row 90
    dc = DeviceCase(case)
    ctx = _ctx(w, True)
    dc.prefill(ctx)  # asserts status OK
    _check(w, dc, case)
    assert np.all(np.isfinite(to_f64(dc.out.bits())[dc.valid_rows()]))
    case.v_new_bits[128 + 60, 1, 0] = np.uint16(0x47C3)  # sequence 1, valid row 60: 99840
    dc2 = DeviceCase(case)
    ctx.prefill(w.cache_lens, w.chunk_lens, dc2.q.t, dc2.k_new.t, dc2.v_new.t, dc2.k_cache.t,
                dc2.v_cache.t, dc2.out.t, dc2.lse)
    assert ctx.sync_status() == cp.E_RANGE
    assert ctx.sync_status() == cp.OK


FULL = [CTX_8K, CTX_32K, CTX_128K, VARLEN]


@pytest.mark.parametrize("staged", [False, True], ids=["bf16cur", "staged"])
@pytest.mark.parametrize("w", FULL, ids=[w.name for w in FULL])
def test_full_size(w, staged):
    """The benchmarked workloads at full size with the fp16 V cache, in the
    launch configuration the benchmark times (staged), and without staging:
    every valid row of one q head per kv head (leader and peer CTAs of a
    pair alternate over the kv heads), and sampled rows of all heads
    (first/last rows of each sequence and q-block edges included), against
    the oracle reading V as stored and as the original bf16 values."""
    case = make_case(w, v_f16=True)
    dc = DeviceCase(case)
    ctx = _ctx(w, staged)
    dc.prefill(ctx)
    out = to_f64(dc.out.bits())
    v = dc.valid_rows()
    heads = heads_per_kv_head(w, pairs=False, seed=w.seed)
    href, _ = case.oracle_heads(heads)
    whole = compare(out[v][:, heads], href[v], f"{w.name} heads {heads}")
    if whole.max_abs_ref < 2:
        assert whole.n_allowance == 0
    samples = sample_rows(w, 48, seed=w.seed)
    ref, ref_lse = case.oracle_rows(samples)
    got = np.stack([out[t, h] for t, h in samples])
    compare(got, ref, w.name)
    # Also against the attention of the original bf16 V values (the fp16
    # conversion is exact for them down to 2^-17).
    ref_bf16, _ = make_case(w).oracle_rows(samples)
    compare(got, ref_bf16, w.name + " vs bf16 V")
    lse = dc.lse.cpu().numpy()
    assert np.max(np.abs(np.array([lse[t, h] for t, h in samples]) - ref_lse)) < 2e-3
    assert np.all(np.isfinite(out[v])), "non-finite output"
    assert dc.guards_intact()
