"""The head pairing modes of the fused prefill against the fp64 oracle.

With an even group size the library pairs adjacent q heads of one kv head.
cpattn_config.pairing picks how: 'mma2' -- the leader CTA of a CTA pair
issues 2-SM MMAs (M = 256) and each CTA stages half of every K/V tile;
'pingpong' -- one CTA holds both heads' query tiles and alternates their
products (HD = 128; 'mma2' at HD = 256); 'none' -- one CTA per unit.  Every
mode must
meet the same bar on cases with several tiles, ragged chunks and an empty
cache, in both P precisions."""
import numpy as np
import pytest

import long_context_chunked_gb300 as cp
from gpu_helpers import DeviceCase, compare, to_f64
from helpers import make_case
from workloads import small

pytestmark = pytest.mark.gpu

MODES = ["mma2", "none", "pingpong"]
CASES = [
    small("pairA", (0, 1000, 129), (300, 130, 256), 320, nq=8, nkv=2, hd=128, shards=4,
          shard_capacity=300, seed=41),
    small("pairB", (2500, 77), (384, 1), 384, nq=4, nkv=1, hd=256, shards=8, seed=42),
    small("pairC", (5000,), (512,), 512, nq=8, nkv=2, hd=256, shards=8, seed=43,
          peaky_frac=0.02),
]


@pytest.mark.parametrize("fast_p", [False, True], ids=["accurate", "fast_p"])
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
@pytest.mark.parametrize("mode", MODES)
def test_pairing_mode_parity(mode, w, fast_p):
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w, fast_p=fast_p, pairing=mode)
    dc.prefill(ctx)
    ref, ref_lse = case.oracle_full()
    v = dc.valid_rows()
    out = to_f64(dc.out.bits())
    if fast_p:
        # bf16 P (an option outside the parity bar): its rounding alone puts
        # the relative RMS near 2.3e-3, so the check is looser.
        compare(out[v], ref[v], f"{mode} {w.name} fast_p", max_abs_bar=2e-2, rel_bar=3.5e-3)
    else:
        compare(out[v], ref[v], f"{mode} {w.name}")
    lse = dc.lse.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lse[v] - ref_lse[v])) < 2e-3, "LSE"
    pad = ~v
    if pad.any():
        assert np.all(dc.out.bits()[pad] == np.uint16(0x7F7F)), "pad rows written"
    assert dc.guards_intact(), "write outside a buffer"


def test_pairing_modes_repeatable():
    """Each mode gives identical bits on a second launch (a race in the
    pair's cross-CTA barriers would show up as run-to-run differences)."""
    w = CASES[2]
    case = make_case(w)
    dc = DeviceCase(case)
    for mode in MODES:
        ctx = cp.Context.for_workload(w, pairing=mode)
        dc.prefill(ctx)
        first = dc.out.bits().copy()
        for _ in range(3):
            dc.prefill(ctx)
            assert np.array_equal(first, dc.out.bits()), mode


ORDER_CASES = [
    # Several rounds of units on the persistent grid, more than one kv head.
    small("ord128", (3000, 1500), (1024, 640), 1024, nq=32, nkv=4, hd=128, shards=8, seed=44),
    small("ord256", (2500,), (1024,), 1024, nq=32, nkv=2, hd=256, shards=8, seed=45),
]


@pytest.mark.parametrize("order", ["longest", "kv_major"])
@pytest.mark.parametrize("w", ORDER_CASES, ids=[w.name for w in ORDER_CASES])
@pytest.mark.parametrize("mode", MODES)
def test_unit_orders(mode, w, order, monkeypatch):
    """Units dealt longest first or kv-head-major (CPATTN_UNIT_ORDER, a test
    override of the cost model's choice): the same parity in every mode."""
    monkeypatch.setenv("CPATTN_UNIT_ORDER", order)
    case = make_case(w)
    dc = DeviceCase(case)
    dc.prefill(cp.Context.for_workload(w, pairing=mode))
    ref, ref_lse = case.oracle_full()
    v = dc.valid_rows()
    compare(to_f64(dc.out.bits())[v], ref[v], f"{mode} {w.name} {order}")
    lse = dc.lse.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lse[v] - ref_lse[v])) < 2e-3, "LSE"
    assert dc.guards_intact()
