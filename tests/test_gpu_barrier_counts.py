"""Barrier accounting of the prefill kernels: every signal matched by its
wait (the PR's Design section names the failure mode -- a signal without
its wait, or a wait without its signal, deadlocks the ring).

The barrier-count build of the library (-DCPATTN_COUNT_BARRIERS) counts,
per CTA, every mbarrier arrival each barrier received and every wait each
role completed (cpattn_set_barrier_counts).  After a launch the counts must
show, for every CTA and barrier:
  * whole phases: arrivals are a multiple of the barrier's arrival count;
  * every full barrier (Q, K/V slot, S, P) observed by its consumer once per
    phase, and every release barrier (Q empty, slot empty) by the producer
    once per phase except the last (nothing refills after it);
  * the phases agree across barriers: one S, one P and one P.V completion per
    tile, slots per tile as the ring layout says, one Q per unit;
  * the softmax's in-order waits for P.V: one per tile from the third on,
    plus one per unit at its epilogue (rescale waits are counted apart);
  * in a CTA pair, the leader's barriers carry both CTAs' arrivals and the
    peer's full barriers none;
and over all CTAs the tiles and units equal what the workload defines.
Cases cross the cache/current boundary, put several units on one CTA and
use both slot parities; they run in every kernel form.  Nothing here can
hang: every wait in the kernels is bounded and the test only reads counts.
"""
import numpy as np
import pytest
import torch

import long_context_chunked_gb300 as cp
from long_context_chunked_gb300 import build as cpbuild
from long_context_chunked_gb300.binding import COUNT_BARS, COUNT_RECORD
from gpu_helpers import DeviceCase
from helpers import make_case
from workloads import small

pytestmark = pytest.mark.gpu

ARRIVE, SOFTMAX, PRODUCER, MMA, RESCALE = range(5)
# Barrier numbers of the kernels (their shared-memory barrier arrays).
QFULL, QEMPTY, SFULL, PFULL, ODONE, DRAIN, SLOTFULL = 0, 1, 2, 4, 6, 8, 9

CASES = [
    # 32 q heads x 7 row blocks: 224 units, two or more per CTA; cache and
    # current tiles in every unit; ragged chunk.
    small("cnt128", (1500, 129), (640, 300), 640, nq=32, nkv=4, hd=128, shards=3, seed=501),
    small("cnt256", (2000, 0), (512, 384), 512, nq=32, nkv=2, hd=256, shards=8, seed=502),
]


@pytest.fixture(scope="module")
def counted_lib():
    return cpbuild.build(variant="counted")


def _form(mode, hd):
    if mode == "pingpong" and hd == 128:
        return "pingpong"
    return "pair2" if mode in ("mma2", "pingpong") else "single"


def _layout(form, hd):
    """(ring slots, slots per tile, arrivals per barrier number)."""
    nslot = 10 if (hd == 256 or form == "pingpong") else 12
    per_tile = {"single": hd // 64 + 128 // (8192 // hd), "pair2": 2 * (hd // 128),
                "pingpong": 4}[form]
    count = np.ones(SLOTFULL + 2 * nslot, dtype=np.int64)
    # HD = 128 (outside the two-tile kernel): one softmax warpgroup per tile.
    takers = 4 if hd == 128 else 8
    if form == "single":
        count[PFULL:PFULL + 2] = 32 * takers
    elif form == "pair2":
        count[PFULL:PFULL + 2] = 2 * takers
        count[QFULL] = 2
        count[SLOTFULL:SLOTFULL + nslot] = 2
    else:
        count[PFULL:PFULL + 2] = 4
    return nslot, per_tile, count


def _run(w, mode, counted_lib, split_tiles=None, fused_write=False, staged=False):
    case = make_case(w, v_f16=staged)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w, pairing=mode, library=counted_lib, v_cache_f16=staged)
    if staged:  # the chunk's V staged in fp16: the every-tile-fp16 kernel form
        ctx._v_stage = torch.empty(ctx.v_staging_bytes(w.num_seqs) // 2, dtype=torch.float16,
                                   device="cuda")
        ctx.set_v_staging(ctx._v_stage)
    if split_tiles is not None:
        need, _ = ctx.splitkv_workspace(w.cache_lens, w.chunk_lens, split_tiles)
        ws = torch.empty(max(need // 4, 64), dtype=torch.float32, device="cuda")
        ctx.set_splitkv(ws, split_tiles)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rec = torch.zeros(sms * COUNT_RECORD, dtype=torch.int32, device="cuda")
    ctx.set_barrier_counts(rec)
    if fused_write:
        ctx.prefill_write_kv(w.cache_lens, w.chunk_lens, dc.q.t, dc.k_new.t, dc.v_new.t,
                             dc.k_cache.t, dc.v_cache.t, dc.out.t, dc.lse)
    else:
        ctx.prefill(w.cache_lens, w.chunk_lens, dc.q.t, dc.k_new.t, dc.v_new.t, dc.k_cache.t,
                    dc.v_cache.t, dc.out.t, dc.lse)
    assert ctx.sync_status() == cp.OK, ctx.last_error()
    counts = rec.cpu().numpy().astype(np.int64).reshape(sms, 5, COUNT_BARS)
    return ctx, counts


def _pv_waits_ok(W, tiles, units, hd, c):
    """The softmax's waits for P.V.  HD = 256: every softmax warp waits in
    order for tile t - 2's product from the CTA's third tile on, and for each
    unit's last product at its epilogue.  HD = 128: only at a unit's
    epilogue, where each warpgroup that took a tile of it waits for its own
    last one (one or two per unit: bounded here, counted exactly over all
    CTAs by the caller); tile t - 2's product is complete once S of tile t
    is, so the tile loop waits for none."""
    got = W[SOFTMAX][ODONE] + W[SOFTMAX][ODONE + 1]
    if hd == 256:
        assert got == 8 * (max(tiles - 2, 0) + units), f"CTA {c}: P.V waits"
        return 0
    assert 4 * units <= got <= 8 * units, f"CTA {c}: P.V waits"
    return got


def _check_cta(c, A, W, form, nslot, per_tile, count, leader=True, hd=256):
    """The per-CTA invariants; returns (tiles, units, epilogue P.V waits) of
    the CTA (the leader's, in a pair)."""
    sw = 4 if hd == 128 else 8  # softmax warps that wait for one S
    nb = SLOTFULL + 2 * nslot
    a = A[:nb]
    assert np.all(a % count == 0), f"CTA {c}: partial phase {a.tolist()} / {count.tolist()}"
    ph = a // count
    SE = SLOTFULL + nslot
    if form == "pair2" and not leader:
        # The peer's full barriers are the leader's: they receive nothing.
        # Its release barriers, S and O get the leader's multicast commits;
        # its own softmax and producer wait on them as the leader's do.
        assert a[QFULL] == 0 and a[PFULL] == 0 and a[PFULL + 1] == 0 and a[DRAIN] == 0
        assert np.all(a[SLOTFULL:SE] == 0), f"CTA {c}"
        assert np.all(W[MMA] == 0), f"CTA {c}: the peer issues no MMA"
        units, tiles = ph[QEMPTY], ph[SFULL] + ph[SFULL + 1]
        for b in (0, 1):
            assert W[SOFTMAX][SFULL + b] == sw * ph[SFULL + b], f"CTA {c}: S waits"
        _pv_waits_ok(W, tiles, units, hd, c)
        assert W[PRODUCER][QEMPTY] == max(units - 1, 0), f"CTA {c}: Q empty"
        assert np.array_equal(W[PRODUCER][SE:SE + nslot], np.maximum(ph[SE:SE + nslot] - 1, 0)), \
            f"CTA {c}: slot-empty waits"
        assert ph[SE:SE + nslot].sum() == tiles * per_tile, f"CTA {c}: slots per tile"
        return None
    units = ph[QFULL]
    assert W[MMA][QFULL] == units, f"CTA {c}: Q waits"
    if form != "pingpong":
        tiles = ph[SFULL] + ph[SFULL + 1]
        for b in (0, 1):
            assert ph[PFULL + b] == ph[SFULL + b] == ph[ODONE + b], f"CTA {c}: S/P/O parity {b}"
            assert W[SOFTMAX][SFULL + b] == sw * ph[SFULL + b], f"CTA {c}: S waits"
            assert W[MMA][PFULL + b] == ph[PFULL + b], f"CTA {c}: P waits"
        epi = _pv_waits_ok(W, tiles, units, hd, c)
        assert W[RESCALE][ODONE] + W[RESCALE][ODONE + 1] <= 8 * tiles
    else:
        tiles = ph[SFULL]
        for q in (0, 1):
            assert ph[SFULL + q] == ph[PFULL + q] == tiles, f"CTA {c}: tile {q} S/P"
            assert ph[ODONE + q] == units, f"CTA {c}: tile {q} O"
            assert W[SOFTMAX][SFULL + q] == 4 * tiles
            assert W[SOFTMAX][ODONE + q] == 4 * units
            assert W[MMA][PFULL + q] == tiles
    assert W[PRODUCER][QEMPTY] == max(units - 1, 0) and ph[QEMPTY] == units, f"CTA {c}: Q empty"
    assert np.array_equal(ph[SLOTFULL:SE], ph[SE:SE + nslot]), f"CTA {c}: slot fill/release"
    assert np.array_equal(W[MMA][SLOTFULL:SE], ph[SLOTFULL:SE]), f"CTA {c}: slot waits"
    assert np.array_equal(W[PRODUCER][SE:SE + nslot], np.maximum(ph[SE:SE + nslot] - 1, 0)), \
        f"CTA {c}: slot-empty waits"
    assert ph[SLOTFULL:SE].sum() == tiles * per_tile, f"CTA {c}: slots per tile"
    assert a[DRAIN] == 1 and W[MMA][DRAIN] == 1, f"CTA {c}: final drain"
    return tiles, units, (epi if form != "pingpong" else 0)


def _check(w, mode, ctx, counts, totals=True):
    form = _form(mode if w.group % 2 == 0 else "none", w.head_dim)
    nslot, per_tile, count = _layout(form, w.head_dim)
    ran = np.nonzero(counts[:, ARRIVE, :].sum(axis=1))[0]
    assert ran.size > 0
    tiles = units = epi = 0
    for c in ran:
        A, W = counts[c, ARRIVE], counts[c]
        if form == "pair2":
            leader = c % 2 == 0
            assert (c ^ 1) in ran, f"CTA {c} ran without its pair"
            r = _check_cta(c, A, W, form, nslot, per_tile, count, leader, w.head_dim)
            if leader:
                # The release barriers are signalled to both CTAs alike.
                peer = counts[c + 1, ARRIVE]
                for i in [QEMPTY, SFULL, SFULL + 1, ODONE, ODONE + 1] + \
                        list(range(SLOTFULL + nslot, SLOTFULL + 2 * nslot)):
                    assert peer[i] == A[i], f"pair {c}: barrier {i}"
                tiles += r[0]
                units += r[1]
                epi += r[2]
        else:
            r = _check_cta(c, A, W, form, nslot, per_tile, count, hd=w.head_dim)
            tiles += r[0]
            units += r[1]
            epi += r[2]
    if totals:
        # Whole walks: a row block (b, qb) has n_cache(b) + qb + 1 tiles; a
        # unit is one q head (single), a head pair (pair2, pingpong).
        per_block = w.num_q_heads // (1 if form == "single" else 2)
        blocks = [(b, qb) for b, c in enumerate(w.chunk_lens) for qb in range(-(-c // 128))]
        n_cache = [len(ctx.cache_walk(L)[0]) for L in w.cache_lens]
        assert units == per_block * len(blocks)
        assert tiles == per_block * sum(n_cache[b] + qb + 1 for b, qb in blocks)
        if w.head_dim == 128 and form != "pingpong":
            # Epilogue waits: one per warp of each warpgroup that took a tile
            # of the unit -- one warpgroup for a one-tile walk, else both.
            assert epi == 4 * per_block * sum(min(n_cache[b] + qb + 1, 2) for b, qb in blocks)
    return tiles, units


@pytest.mark.parametrize("order", ["longest", "kv_major"])
@pytest.mark.parametrize("mode", ["mma2", "none", "pingpong"])
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_barrier_counts_balance(w, mode, order, counted_lib, monkeypatch):
    monkeypatch.setenv("CPATTN_UNIT_ORDER", order)
    ctx, counts = _run(w, mode, counted_lib)
    _check(w, mode, ctx, counts)


@pytest.mark.parametrize("mode", ["mma2", "none", "pingpong"])
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_barrier_counts_staged_v(w, mode, counted_lib):
    """The every-tile-fp16 form (the chunk's V staged, its prefill a
    programmatic dependent of the staging) keeps the same balance."""
    ctx, counts = _run(w, mode, counted_lib, staged=True)
    _check(w, mode, ctx, counts)


def test_barrier_counts_fused_write(counted_lib):
    ctx, counts = _run(CASES[0], "mma2", counted_lib, fused_write=True)
    _check(CASES[0], "mma2", ctx, counts)


@pytest.mark.parametrize("mode", ["mma2", "none"])
def test_barrier_counts_split_pieces(mode, counted_lib):
    """Split-KV pieces start mid-walk: the tiles over all pieces are the
    whole walks' tiles, and every piece loads its Q once."""
    w = CASES[1]
    ctx, counts = _run(w, mode, counted_lib, split_tiles=4)
    tiles, units = _check(w, mode, ctx, counts, totals=False)
    per_block = w.num_q_heads // (2 if mode == "mma2" else 1)
    blocks = [(b, qb) for b, c in enumerate(w.chunk_lens) for qb in range(-(-c // 128))]
    n_cache = [len(ctx.cache_walk(L)[0]) for L in w.cache_lens]
    assert tiles == per_block * sum(n_cache[b] + qb + 1 for b, qb in blocks)
    assert units > per_block * len(blocks)


def test_barrier_counts_gqa_packed_decode(counted_lib):
    w = small("cntdec", (3000, 700), (1, 3), 64, nq=8, nkv=2, hd=256, shards=8, seed=503)
    ctx, counts = _run(w, "mma2", counted_lib)
    _check(w, "none", ctx, counts, totals=False)  # packed units run unpaired


def test_release_build_leaves_counts_alone():
    """The release library refuses counting, and its kernels take no
    counting path."""
    w = CASES[0]
    ctx = cp.Context.for_workload(w)
    rec = torch.zeros(COUNT_RECORD, dtype=torch.int32, device="cuda")
    with pytest.raises(cp.CpattnError) as e:
        ctx.set_barrier_counts(rec)
    assert e.value.status == cp.E_UNSUPPORTED
