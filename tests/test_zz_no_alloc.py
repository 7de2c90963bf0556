"""The allocation-free prefill entry point against the fp64 oracle and
against the context-based entry point.

cpattn_prefill_noalloc serves callers that cannot allocate device memory
(code running while a pooled or custom allocator owns the device, regions
where cudaMalloc/cudaFree are forbidden or would synchronise, embedders that
only pass pointers): it keeps the kernel's status word in a static device
array instead of a cudaMalloc'd one.  Two calls in a row must each meet the
parity bar of the other GPU tests against the oracle, and agree with
cpattn_prefill's output within that bar, in every kernel instantiation the
entry point launches (both head dims, both P precisions, bf16 and fp16 V
caches), with and without the LSE output.  This file is collected last.
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


def _bars(fast_p):
    # bf16 P (fast_p, an option outside the parity bar) takes the looser bar
    # its own tests use; every other form takes the standard one.
    return dict(max_abs_bar=2e-2, rel_bar=3.5e-3) if fast_p else {}


@pytest.mark.parametrize("v_f16", [False, True], ids=["bf16_v", "f16_v"])
@pytest.mark.parametrize("fast_p", [False, True], ids=["accurate", "fast_p"])
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_noalloc_parity(w, fast_p, v_f16):
    case = make_case(w, v_f16=v_f16)
    dc = DeviceCase(case)
    ref, ref_lse = case.oracle_full()
    v = dc.valid_rows()
    # The context-based entry point on the same inputs.
    ctx = cp.Context.for_workload(w, fast_p=fast_p, v_cache_f16=v_f16)
    dc.prefill(ctx)
    ctx_out = to_f64(dc.out.bits())
    cfg = binding.Config(w.num_q_heads, w.num_kv_heads, w.head_dim, w.shards, w.shard_capacity,
                         w.chunk, w.scale, int(fast_p), int(v_f16), 0, 0)
    for call in range(2):
        out = Guarded((w.tokens, w.num_q_heads, w.head_dim))
        with_lse = call == 0  # the second call passes lse = NULL
        lse = torch.full((w.tokens, w.num_q_heads), float("nan"), dtype=torch.float32,
                         device="cuda") if with_lse else None
        st = binding.prefill_noalloc(cfg, w.cache_lens, w.chunk_lens, dc.q.t, dc.k_new.t,
                                     dc.v_new.t, dc.k_cache.t, dc.v_cache.t, out.t, lse)
        assert st == cp.OK, f"call {call}: status {st}"
        torch.cuda.synchronize()
        got = to_f64(out.bits())
        compare(got[v], ref[v], f"{w.name} call {call} vs oracle", **_bars(fast_p))
        compare(got[v], ctx_out[v], f"{w.name} call {call} vs cpattn_prefill", **_bars(fast_p))
        if with_lse:
            assert np.max(np.abs(lse.cpu().numpy()[v] - ref_lse[v])) < 2e-3
        pad = ~v
        if pad.any():
            assert np.all(out.bits()[pad] == np.uint16(0x7F7F)), "pad rows written"
        assert out.guards_intact(), "write outside the output"
    assert dc.guards_intact()


def test_noalloc_rejects_sizes_beyond_tables():
    w = TINY
    cfg = binding.Config(w.num_q_heads, w.num_kv_heads, w.head_dim, w.shards, w.shard_capacity,
                         w.chunk, w.scale, 0, 0, 0, 0)
    A = 256
    too_many = [0] * (binding.MAX_SEQS + 1)
    assert binding.prefill_noalloc(cfg, too_many, [1] * len(too_many), A, A, A, A, A, A,
                                   stream=0) == cp.E_UNSUPPORTED
    assert binding.prefill_noalloc(cfg, [0], [w.chunk + 1], A, A, A, A, A, A,
                                   stream=0) == cp.E_INVALID
