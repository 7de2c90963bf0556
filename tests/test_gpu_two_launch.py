"""The removed two-launch variant (cache-only launch + current-only launch +
LSE merge) against the oracle, and against the fused kernel: the PR's
Summary section removed it as slower, not as different."""
import numpy as np
import pytest
import torch

import long_context_chunked_gb300 as cp
from gpu_helpers import DeviceCase, Guarded, compare, to_f64
from helpers import make_case, sample_rows
from workloads import CTX_32K, small

pytestmark = pytest.mark.gpu

CASES = [
    small("tl_a", (0, 300, 129), (200, 256, 1), 256, nq=8, nkv=2, hd=128, shards=2, seed=61),
    small("tl_b", (1000, 0), (130, 64), 256, nq=4, nkv=1, hd=256, shards=4, shard_capacity=300,
          seed=62),
    small("tl_c", (777,), (129,), 192, nq=6, nkv=3, hd=256, shards=8, seed=63),
]


def _two_launch(dc, ctx, w):
    ws = torch.empty(ctx.two_launch_workspace(w.num_seqs), dtype=torch.uint8, device="cuda")
    out = Guarded((w.tokens, w.num_q_heads, w.head_dim))
    lse = torch.full((w.tokens, w.num_q_heads), float("nan"), dtype=torch.float32, device="cuda")
    ctx.prefill_two_launch(w.cache_lens, w.chunk_lens, dc.q.t, dc.k_new.t, dc.v_new.t,
                           dc.k_cache.t, dc.v_cache.t, out.t, ws, lse)
    assert ctx.sync_status() == 0, ctx.last_error()
    assert out.guards_intact()
    return to_f64(out.bits()), lse.cpu().numpy()


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_two_launch_matches_oracle_and_fused(w):
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    dc.prefill(ctx)
    fused = to_f64(dc.out.bits())
    got, lse = _two_launch(dc, ctx, w)
    ref, ref_lse = case.oracle_full()
    v = dc.valid_rows()
    compare(got[v], ref[v], f"{w.name} two-launch vs oracle")
    assert np.max(np.abs(lse[v] - ref_lse[v])) < 2e-3
    compare(got[v], fused[v], f"{w.name} two-launch vs fused")


def test_two_launch_32k_sampled():
    w = CTX_32K
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    got, _ = _two_launch(dc, ctx, w)
    samples = sample_rows(w, 32, seed=5)
    ref, _ = case.oracle_rows(samples)
    compare(np.stack([got[t, h] for t, h in samples]), ref, "32k two-launch")
