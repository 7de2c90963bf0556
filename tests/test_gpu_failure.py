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


@pytest.mark.parametrize("kind", ["unpaired", "packed_split"])
def test_bounded_wait_other_kernels(kind):
    """The same check on the unpaired kernel (group size 1, as GQA-packed
    launches run) and on a split-KV launch of packed decode rows: the expired
    wait is reported, the merge of the incomplete pieces does not hang, and
    the context then computes correctly."""
    import torch
    if kind == "unpaired":
        w = small("failu", (300,), (200,), 256, nq=3, nkv=3, hd=128, shards=2, seed=95)
    else:
        w = small("failp", (20000,), (1,), 64, nq=16, nkv=2, hd=256, shards=8, seed=96)
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    if kind == "packed_split":
        need, _ = ctx.splitkv_workspace(w.cache_lens, w.chunk_lens, 8)
        ws = torch.empty(max(need // 4, 64), dtype=torch.float32, device="cuda")
        ctx.set_splitkv(ws, 8)
    ctx.set_fault_injection(1, timeout_ms=50)
    ctx.prefill(w.cache_lens, w.chunk_lens, dc.q.t, dc.k_new.t, dc.v_new.t, dc.k_cache.t,
                dc.v_cache.t, dc.out.t)
    assert ctx.sync_status() == cp.E_TIMEOUT
    assert ctx.sync_status() == cp.OK
    ctx.set_fault_injection(0, 0)
    dc.prefill(ctx)
    ref, _ = case.oracle_full()
    v = dc.valid_rows()
    compare(to_f64(dc.out.bits())[v], ref[v], f"{kind} after timeout")
