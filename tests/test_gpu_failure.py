"""Failure detection without a GPU fault: a test-only hook makes one thread of
the first CTA skip one internal mbarrier arrival.  Every wait in the kernel is
bounded, so that CTA's roles give up after the (short) limit, drain their
copies and MMAs, free TMEM and return; the host then reads E_TIMEOUT from the
status word, and the same context computes correctly afterwards."""
import numpy as np
import pytest

import long_context_chunked_gb300 as cp
from gpu_helpers import DeviceCase, compare, to_f64
from helpers import make_case
from workloads import small

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hd", [128, 256])
def test_bounded_wait_reports_timeout_and_context_survives(hd):
    w = small(f"fail{hd}", (300,), (256,), 256, nq=4, nkv=2, hd=hd, shards=2, seed=90 + hd)
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    ctx.set_fault_injection(1, timeout_ms=50)
    ctx.prefill(w.cache_lens, w.chunk_lens, dc.q.t, dc.k_new.t, dc.v_new.t, dc.k_cache.t,
                dc.v_cache.t, dc.out.t)
    assert ctx.sync_status() == cp.E_TIMEOUT
    assert "site" in ctx.last_error()
    assert ctx.sync_status() == cp.OK  # the status word was cleared
    ctx.set_fault_injection(0, 0)
    dc.prefill(ctx)
    ref, _ = case.oracle_full()
    v = dc.valid_rows()
    compare(to_f64(dc.out.bits())[v], ref[v], "after timeout")
