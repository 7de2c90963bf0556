"""Fused prefill on the GPU against the fp64 oracle.

Small cases compare every valid output element; the four full-size
workloads, in the launch configuration the benchmark uses, compare every
valid row of whole q heads (an adjacent pair per kv head -- the two heads
one CTA pair computes -- at 8k, 32k and varlen, one head per kv head at
128k), seeded sampled rows of all heads (first/last rows of each sequence
and q block edges included), and whole-output properties.  Bar: max |diff| <= 1e-2 and relative RMS
<= 2e-3.  Cache holes hold large finite poison; guard bands around every
buffer must survive."""
import numpy as np
import pytest
import torch

import oracle
import long_context_chunked_gb300 as cp
from gpu_helpers import DeviceCase, compare, to_f64
from helpers import POISON_BITS, heads_per_kv_head, make_case, sample_rows
from workloads import ALL, CTX_8K, CTX_32K, CTX_128K, TINY, VARLEN, small

pytestmark = pytest.mark.gpu


def _full_parity(w, with_lse=True):
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    dc.prefill(ctx, with_lse)
    ref, ref_lse = case.oracle_full()
    v = dc.valid_rows()
    out = to_f64(dc.out.bits())
    res = compare(out[v], ref[v], w.name)
    if with_lse:
        lse = dc.lse.cpu().numpy().astype(np.float64)
        assert np.max(np.abs(lse[v] - ref_lse[v])) < 2e-3, "LSE"
    # pad rows are never written
    pad = ~v
    if pad.any():
        assert np.all(dc.out.bits()[pad] == np.uint16(0x7F7F)), "pad rows written"
    assert dc.guards_intact(), "write outside a buffer"
    return res


def test_tiny_full():
    _full_parity(TINY)


EDGE = []
for hd in (128, 256):
    for L in (0, 1, 127, 128, 129):
        for c in (1, 127, 128, 129):
            EDGE.append(small(f"L{L}c{c}h{hd}", (L,), (c,), 192, nq=4, nkv=2, hd=hd, shards=2,
                              seed=L * 1000 + c + hd))
EDGE += [
    # P in {1, 4, 8}; several tiles per shard; S not a multiple of the tile height
    small("p1", (300,), (200,), 256, nq=2, nkv=1, hd=128, shards=1, seed=7),
    small("p4", (1000,), (130,), 256, nq=8, nkv=2, hd=256, shards=4, shard_capacity=300, seed=8),
    small("p8", (2000,), (64,), 128, nq=4, nkv=4, hd=128, shards=8, shard_capacity=333, seed=9),
    small("tinyS", (500,), (40,), 64, nq=2, nkv=1, hd=128, shards=8, shard_capacity=70, seed=10),
    # several sequences with empty, ragged and full chunks
    small("multi", (0, 50, 700, 129, 256), (300, 0, 17, 256, 128), 300, nq=8, nkv=2, hd=128,
          shards=4, seed=11),
    small("multi256", (1, 999, 128), (5, 384, 255), 384, nq=4, nkv=1, hd=256, shards=2,
          seed=12),
    small("mha", (333,), (222,), 256, nq=3, nkv=3, hd=128, shards=3, seed=13),
    small("peaky", (3000,), (500,), 512, nq=8, nkv=2, hd=256, shards=8, seed=14, peaky_frac=0.05),
]


@pytest.mark.parametrize("w", EDGE, ids=[w.name for w in EDGE])
def test_edges_full(w):
    _full_parity(w)


FULL = [CTX_8K, CTX_32K, CTX_128K, VARLEN]


@pytest.fixture(scope="module")
def full_runs():
    return {}


@pytest.mark.parametrize("w", FULL, ids=[w.name for w in FULL])
def test_full_size(w, full_runs):
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    dc.prefill(ctx)
    out = to_f64(dc.out.bits())
    v = dc.valid_rows()
    # Whole q heads: every valid row of every sequence.
    heads = heads_per_kv_head(w, pairs=w is not CTX_128K)
    href, href_lse = case.oracle_heads(heads)
    whole = compare(out[v][:, heads], href[v], f"{w.name} heads {heads}")
    if whole.max_abs_ref < 2:
        assert whole.n_allowance == 0
    lse_all = dc.lse.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lse_all[v][:, heads] - href_lse[v])) < 2e-3, "LSE (whole heads)"
    # Sampled rows of every head.
    samples = sample_rows(w, 48, seed=w.seed)
    ref, ref_lse = case.oracle_rows(samples)
    got = np.stack([out[t, h] for t, h in samples])
    max_abs, rel = compare(got, ref, w.name)[:2]
    lse = dc.lse.cpu().numpy()
    assert np.max(np.abs(np.array([lse[t, h] for t, h in samples]) - ref_lse)) < 2e-3
    assert np.all(np.isfinite(out[v])), "non-finite output"
    assert np.all(np.abs(out[v]) < 16), "output outside the convex hull of V"
    assert dc.guards_intact()
    # Negative control: the same samples against an oracle given different
    # cache contents must miss by far more than the passing error.
    bad = make_case(w.with_(seed=w.seed + 1000))
    bad.q_bits, bad.k_new_bits, bad.v_new_bits = case.q_bits, case.k_new_bits, case.v_new_bits
    nref, _ = bad.oracle_rows(samples)
    neg = float(np.max(np.abs(got - nref)))
    if sum(w.cache_lens) > 0:
        assert neg >= 50 * max(max_abs, 1e-4), f"negative control {neg:.3e} vs pass {max_abs:.3e}"
    full_runs[w.name] = (max_abs, rel, neg)


def test_equal_keys_prefix_mean():
    """All keys equal: every row is the plain mean of its visible values --
    pins the causal diagonal, the cache visibility and the shard walk."""
    w = small("eqk", (700, 0), (300, 256), 320, nq=4, nkv=2, hd=128, shards=4,
              shard_capacity=260, seed=21)
    case = make_case(w)
    kvec = case.k_new_bits[0, :, :].copy()
    case.k_new_bits[...] = kvec[None]
    case.k_cache_bits[...] = kvec[None, :, None, None, :]
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    dc.prefill(ctx)
    out = to_f64(dc.out.bits())
    vn = case.f64("v_new")
    G = w.group
    for b, (L, c) in enumerate(zip(w.cache_lens, w.chunk_lens)):
        vc = oracle.read_logical(case.f64("v_cache"), b, L)
        for h in range(w.num_q_heads):
            g = h // G
            tot = vc[:, g].sum(axis=0) if L else np.zeros(w.head_dim)
            run = np.cumsum(vn[b * w.chunk: b * w.chunk + c, g], axis=0)
            ref = (tot[None] + run) / (L + np.arange(1, c + 1))[:, None]
            compare(out[b * w.chunk: b * w.chunk + c, h], ref, f"equal keys b={b} h={h}")


def test_repeatable_and_write_order_independent():
    """Two launches give identical bits; running write_kv first changes nothing
    (prefill reads only cache rows of tokens < L)."""
    w = small("rep", (900,), (256,), 256, nq=8, nkv=2, hd=256, shards=4, seed=31)
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    dc.prefill(ctx)
    first = dc.out.bits().copy()
    ctx.write_kv(w.cache_lens, w.chunk_lens, dc.k_new.t, dc.v_new.t, dc.k_cache.t, dc.v_cache.t)
    dc.prefill(ctx)
    assert np.array_equal(first, dc.out.bits())


@pytest.mark.parametrize("hd,nq,nkv,mode", [(128, 4, 2, "mma2"), (256, 8, 2, "mma2"),
                                             (128, 3, 3, "mma2"), (128, 4, 2, "pingpong")])
def test_rescale_on_every_tile(hd, nq, nkv, mode, monkeypatch):
    """Keys constant along each row, stepping up by 0.5 per tile in walk
    order (cache flat rows, then the chunk's tiles), queries all ones: every
    tile's row max exceeds the running max by sqrt(HD) * 0.5 * log2(e) > 8, so
    the lazy rescale of O -- and its wait for the previous tile's P.V --
    runs on every tile of every unit, in the paired, unpaired and two-tile
    kernels."""
    monkeypatch.setenv("CPATTN_PAIRING", mode)
    w = small(f"resc{hd}", (1500, 300), (300, 200), 320, nq=nq, nkv=nkv, hd=hd, shards=3,
              shard_capacity=700, seed=41 + hd)
    case = make_case(w)
    one = np.uint16(0x3F80)
    case.q_bits[...] = one

    def bf16_of(x):  # exact: multiples of 0.5 below 256
        return oracle.bf16_bits(torch.tensor([float(x)]).to(torch.bfloat16))[0]

    kc = case.k_cache_bits  # [B, NKV, P, S, HD]
    B, NKV, P, S, HD = kc.shape
    top = 0
    for b in range(B):
        for s in range(P):
            for r in range(S):
                f = s * S + r  # flat row of the (sequence, kv head) walk
                kc[b, :, s, r, :] = bf16_of(0.5 * (f // 128))
        top = max(top, (P * S) // 128 + 1)
    for b, c in enumerate(w.chunk_lens):
        for i in range(c):
            case.k_new_bits[b * w.chunk + i, :, :] = bf16_of(0.5 * (top + i // 128))
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    dc.prefill(ctx)
    ref, ref_lse = case.oracle_full()
    v = dc.valid_rows()
    compare(to_f64(dc.out.bits())[v], ref[v], f"rescale every tile, HD={hd}")
    lse = dc.lse.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lse[v] - ref_lse[v])) / max(1.0, np.max(np.abs(ref_lse[v]))) < 2e-3
    assert dc.guards_intact()
