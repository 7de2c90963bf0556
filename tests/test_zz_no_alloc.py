"""The allocation-free prefill entry point against the context-based one.

cpattn_prefill_noalloc serves callers that cannot allocate device memory
(pooled/custom allocators, regions where cudaMalloc is forbidden): it keeps
the kernel's status word in a static device array instead of a cudaMalloc'd
one.  Two calls in a row must each reproduce cpattn_prefill's output within
the parity tolerance of the other GPU tests.  This file is collected last.
"""
import numpy as np
import pytest
import torch

import long_context_chunked_gb300 as cp
from long_context_chunked_gb300 import binding
from gpu_helpers import DeviceCase, Guarded, compare, to_f64
from helpers import make_case
from workloads import TINY, small

pytestmark = pytest.mark.gpu

CASES = [TINY, small("na256", (0, 700, 129), (300, 256, 5), 320, nq=8, nkv=2, hd=256,
                     shards=4, seed=77)]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_noalloc_matches_context_path(w):
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    dc.prefill(ctx)
    ref = to_f64(dc.out.bits())
    ref_lse = dc.lse.cpu().numpy()
    v = dc.valid_rows()
    cfg = binding.Config(w.num_q_heads, w.num_kv_heads, w.head_dim, w.shards, w.shard_capacity,
                         w.chunk, w.scale, 0)
    for call in range(2):
        out = Guarded((w.tokens, w.num_q_heads, w.head_dim))
        lse = torch.full((w.tokens, w.num_q_heads), float("nan"), dtype=torch.float32,
                         device="cuda")
        st = binding.prefill_noalloc(cfg, w.cache_lens, w.chunk_lens, dc.q.t, dc.k_new.t,
                                     dc.v_new.t, dc.k_cache.t, dc.v_cache.t, out.t, lse)
        assert st == cp.OK, f"call {call}: status {st}"
        torch.cuda.synchronize()
        got = to_f64(out.bits())
        compare(got[v], ref[v], f"{w.name} call {call}")
        assert np.max(np.abs(lse.cpu().numpy()[v] - ref_lse[v])) < 2e-3
        assert out.guards_intact()


def test_noalloc_rejects_sizes_beyond_tables():
    w = TINY
    cfg = binding.Config(w.num_q_heads, w.num_kv_heads, w.head_dim, w.shards, w.shard_capacity,
                         w.chunk, w.scale, 0)
    A = 256
    too_many = [0] * (binding.MAX_SEQS + 1)
    assert binding.prefill_noalloc(cfg, too_many, [1] * len(too_many), A, A, A, A, A, A,
                                   stream=0) == cp.E_UNSUPPORTED
    assert binding.prefill_noalloc(cfg, [0], [w.chunk + 1], A, A, A, A, A, A,
                                   stream=0) == cp.E_INVALID
