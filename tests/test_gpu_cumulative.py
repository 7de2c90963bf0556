"""A whole chunked prefill, chunk after chunk, against the fp64 oracle (the
PR's per-request cumulative prefill, Performance section).

Each step writes the chunk into the striped caches and prefills it against
everything the earlier steps left there: cpattn_write_kv then cpattn_prefill
(or both in one launch, cpattn_prefill_write_kv), the cache length growing
by the earlier chunks.  The oracle keeps its own caches, applying its own
scatter step by step, and computes every step's attention from them.  Every
step's output is compared at the standard bar; the caches after the last
step must equal the oracle's bit for bit over the whole buffers, and no
write may leave them.  The shard count divides neither the chunk nor the
requests, so shard fill is unequal at every step; one sequence brings
ragged and empty chunks."""
import numpy as np
import pytest
import torch

import oracle
import long_context_chunked_gb300 as cp
from gpu_helpers import Guarded, compare, to_f64
from workloads import generate_request, request

pytestmark = pytest.mark.gpu

REQUESTS = [
    request("cum128", [(200, 200), (200, 37), (200, 0), (200, 200), (200, 129)], 200, nq=4,
            nkv=2, hd=128, shards=3, seed=301),
    request("cum256", [(200, 128), (200, 200), (200, 1), (200, 200), (150, 200)], 200, nq=8,
            nkv=2, hd=256, shards=3, seed=302),
]


def _valid(w):
    m = np.zeros(w.tokens, dtype=bool)
    for b, c in enumerate(w.chunk_lens):
        m[b * w.chunk: b * w.chunk + c] = True
    return m


@pytest.mark.parametrize("fused", [False, True], ids=["write_then_prefill", "fused_write"])
@pytest.mark.parametrize("v_f16,staged", [(False, False), (True, False), (True, True)],
                         ids=["bf16_v", "f16_v", "f16_v_staged"])
@pytest.mark.parametrize("r", REQUESTS, ids=[r.name for r in REQUESTS])
def test_cumulative_request(r, v_f16, staged, fused):
    steps = generate_request(r)
    shape = (r.num_seqs, r.num_kv_heads, r.shards, r.shard_capacity, r.head_dim)
    # Both sides start from the same caches (finite fill, the chunk rows
    # arrive through the writes).
    kc_ref = np.full(shape, 0x3F00, dtype=np.uint16)   # bf16 0.5
    vc_ref = np.full(shape, 0x3800 if v_f16 else 0x3F00, dtype=np.uint16)  # 0.5
    kc = Guarded(shape, kc_ref)
    vc = Guarded(shape, vc_ref, dtype=torch.float16 if v_f16 else torch.bfloat16)
    ctx = cp.Context(r.num_q_heads, r.num_kv_heads, r.head_dim, r.shards, r.shard_capacity,
                     r.chunk, 0.0, False, v_f16)
    if staged:  # the chunk's V staged in fp16: every tile takes fp16 P
        stage = torch.empty(ctx.v_staging_bytes(r.num_seqs) // 2, dtype=torch.float16,
                            device="cuda")
        ctx.set_v_staging(stage)
    vconv = oracle.f16_bits_to_f64 if v_f16 else oracle.bits_to_f64
    for k, inp in enumerate(steps):
        w = r.step(k)
        q_bits, kn_bits, vn_bits = (oracle.bf16_bits(x) for x in (inp.q, inp.k_new, inp.v_new))
        q, kn, vn = Guarded(q_bits.shape, q_bits), Guarded(kn_bits.shape, kn_bits), \
            Guarded(vn_bits.shape, vn_bits)
        out = Guarded((w.tokens, w.num_q_heads, w.head_dim))
        if fused:
            ctx.prefill_write_kv(w.cache_lens, w.chunk_lens, q.t, kn.t, vn.t, kc.t, vc.t, out.t)
        else:
            ctx.write_kv(w.cache_lens, w.chunk_lens, kn.t, vn.t, kc.t, vc.t)
            ctx.prefill(w.cache_lens, w.chunk_lens, q.t, kn.t, vn.t, kc.t, vc.t, out.t)
        assert ctx.sync_status() == cp.OK, ctx.last_error()
        # Oracle: attention over its own caches as they stand before this
        # step's write (the prefill reads only tokens < L_b), then its write.
        ref, _ = oracle.attend_ref(q_bits, kn_bits, vn_bits, oracle.bits_to_f64(kc_ref),
                                   vconv(vc_ref), w.cache_lens, w.chunk_lens, w.chunk, w.scale)
        oracle.write_kv_ref(kc_ref, vc_ref, kn_bits, vn_bits, w.cache_lens, w.chunk_lens,
                            w.chunk, v_f16=v_f16)
        v = _valid(w)
        if v.any():
            compare(to_f64(out.bits())[v], ref[v], f"{r.name} step {k} (L={w.cache_lens})")
        assert np.all(out.bits()[~v] == np.uint16(0x7F7F)), "pad rows written"
        assert out.guards_intact() and q.guards_intact()
    assert np.array_equal(kc.bits(), kc_ref), "K cache differs from the oracle's writes"
    assert np.array_equal(vc.bits(), vc_ref), "V cache differs from the oracle's writes"
    assert kc.guards_intact() and vc.guards_intact(), "write outside a cache"
