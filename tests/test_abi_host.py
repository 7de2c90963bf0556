"""Host-side checks of the C-ABI library: loads, exports every declared symbol,
validates arguments before any launch, and walks the cache exactly over the
filled rows of the striped layout.  No GPU needed."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import long_context_chunked_gb300 as cp
from long_context_chunked_gb300 import build as cpbuild
from workloads import ALL

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cpbuild.build()
    return cp.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "cpattn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cpattn_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert len(names) >= 9
    assert sorted(cp.EXPORTS) == names
    for n in names:
        assert hasattr(lib, n), n


def test_every_export_has_a_typed_binding(lib):
    """ctypes defaults to 32-bit int arguments: an entry point called without
    argtypes would truncate device pointers.  Every symbol must be typed."""
    for n in cp.EXPORTS:
        fn = getattr(lib, n)
        if n != "cpattn_destroy":
            assert fn.restype is not None, n
        assert fn.argtypes is not None and len(fn.argtypes) >= 1, n


def test_status_strings(lib):
    for s in range(6):
        assert lib.cpattn_status_string(s)
    assert lib.cpattn_status_string(99) == b"unknown status"


@pytest.mark.parametrize("cfg,status", [
    ((4, 3, 128, 2, 8, 8), cp.E_INVALID),      # NQ % NKV
    ((4, 2, 64, 2, 8, 8), cp.E_UNSUPPORTED),   # HD
    ((4, 2, 128, 0, 8, 8), cp.E_INVALID),      # P
    ((4, 2, 128, 2, 0, 8), cp.E_INVALID),      # S
    ((4, 2, 128, 2, 8, 0), cp.E_INVALID),      # C
])
def test_create_rejects(lib, cfg, status):
    with pytest.raises(cp.CpattnError) as e:
        cp.Context(*cfg)
    assert e.value.status == status


@pytest.mark.parametrize("field,value", [("fast_p", 2), ("v_cache_f16", -1), ("pairing", 3),
                                         ("pairing", -1), ("gqa_packing", 2)])
def test_create_rejects_config_fields(lib, field, value):
    """Every enumerated field of cpattn_config is range-checked at create, and
    by the allocation-free prefill before anything runs."""
    cfg = cp.binding.Config(8, 2, 128, 2, 64, 32, 0.0, 0, 0, 0, 0)
    setattr(cfg, field, value)
    h = ctypes.c_void_p()
    assert lib.cpattn_create(ctypes.byref(cfg), ctypes.byref(h)) == cp.E_INVALID
    assert not h.value
    A = 256
    assert cp.binding.prefill_noalloc(cfg, [0], [1], A, A, A, A, A, A, stream=0) == cp.E_INVALID


def test_too_many_q_heads_unsupported(lib):
    """More than 65535 q heads would overflow the kernel's unit count: refused
    by create and by the allocation-free prefill alike."""
    cfg = cp.binding.Config(65536, 1, 128, 2, 64, 32, 0.0, 0, 0, 0, 0)
    h = ctypes.c_void_p()
    assert lib.cpattn_create(ctypes.byref(cfg), ctypes.byref(h)) == cp.E_UNSUPPORTED
    A = 256
    assert cp.binding.prefill_noalloc(cfg, [0], [1], A, A, A, A, A, A,
                                      stream=0) == cp.E_UNSUPPORTED


def test_pairing_and_packing_from_config(lib):
    """The kernel form is a configuration field: pairing "pingpong" plans one
    executor per SM at HD = 128 (more split pieces than 2-SM pairs), and
    gqa_packing off leaves a decode step unpacked."""
    a = cp.Context(8, 2, 128, 8, 8000, 128, pairing="mma2")
    b = cp.Context(8, 2, 128, 8, 8000, 128, pairing="pingpong")
    assert b.splitkv_workspace([60000], [100], 0)[1] > a.splitkv_workspace([60000], [100], 0)[1]
    on = cp.Context(32, 2, 256, 8, 1000, 64)
    off = cp.Context(32, 2, 256, 8, 1000, 64, gqa_packing=False)
    assert on.splitkv_workspace([5000, 5000], [64, 1], 1 << 20)[1] == 8 + 1
    assert off.splitkv_workspace([5000, 5000], [64, 1], 1 << 20)[1] == 2


@pytest.mark.parametrize("value,ok", [("mma2", True), ("none", True), ("pingpong", True),
                                      ("multicast", False), ("both", False), ("", False)])
def test_pairing_override_from_environment(lib, monkeypatch, value, ok):
    """CPATTN_PAIRING (a test override of cpattn_config.pairing) is read at
    create; an unknown value is rejected there rather than silently running
    another kernel."""
    monkeypatch.setenv("CPATTN_PAIRING", value)
    if ok:
        cp.Context(8, 2, 128, 2, 64, 32).close()
    else:
        with pytest.raises(cp.CpattnError) as e:
            cp.Context(8, 2, 128, 2, 64, 32)
        assert e.value.status == cp.E_INVALID


@pytest.mark.parametrize("value,ok", [("auto", True), ("off", True), ("on", False)])
def test_gqa_packing_override_from_environment(lib, monkeypatch, value, ok):
    monkeypatch.setenv("CPATTN_GQA_PACKING", value)
    if ok:
        # The override wins over the configuration field.
        ctx = cp.Context(32, 2, 256, 8, 1000, 64, gqa_packing=(value == "off"))
        # A decode step is packed (one 8-token block) unless packing is off.
        _, blocks = ctx.splitkv_workspace([5000], [1], 1 << 20)
        assert blocks == 1
        _, blocks = ctx.splitkv_workspace([5000, 5000], [64, 1], 1 << 20)
        assert blocks == (8 + 1 if value == "auto" else 2)
    else:
        with pytest.raises(cp.CpattnError) as e:
            cp.Context(32, 2, 256, 8, 1000, 64)
        assert e.value.status == cp.E_INVALID


@pytest.mark.parametrize("value,ok", [("auto", True), ("longest", True), ("kv_major", True),
                                      ("kv", False)])
def test_unit_order_override_from_environment(lib, monkeypatch, value, ok):
    monkeypatch.setenv("CPATTN_UNIT_ORDER", value)
    if ok:
        cp.Context(8, 2, 128, 2, 64, 32).close()
    else:
        with pytest.raises(cp.CpattnError) as e:
            cp.Context(8, 2, 128, 2, 64, 32)
        assert e.value.status == cp.E_INVALID


def test_no_multicast_tma_load_in_the_sources():
    """The library may be launched on several GPUs (one replica per GPU), so
    no TMA load in it may use cluster multicast; mbarrier signals
    (tcgen05.commit ... multicast::cluster) are not loads and are allowed."""
    d = os.path.join(ROOT, "long_context_chunked_gb300", "csrc")
    for name in sorted(os.listdir(d)) + ["../../include/cpattn.h"]:
        text = open(os.path.join(d, name)).read()
        assert not re.search(r"cp\.async\.bulk[^;]*multicast", text), name


def test_barrier_counts_need_the_count_build(lib):
    """The release library refuses barrier counting; the count build accepts
    a record buffer and rejects a misaligned one."""
    ctx = cp.Context(8, 2, 128, 2, 64, 32)
    assert ctx.lib.cpattn_set_barrier_counts(ctx._h, 4096, 4096) == cp.E_UNSUPPORTED
    assert ctx.lib.cpattn_set_barrier_counts(ctx._h, None, 0) == cp.E_UNSUPPORTED


def test_prefill_and_write_validation(lib):
    ctx = cp.Context(8, 2, 128, 2, 64, 32)
    A = 256  # a 16-byte-aligned stand-in pointer; nothing is launched
    good = dict(q=A, k_new=A, v_new=A, k_cache=A, v_cache=A, out=A)

    def pf(cl, ch, **kw):
        args = dict(good, **kw)
        return ctx.prefill_raw(cl, ch, args["q"], args["k_new"], args["v_new"], args["k_cache"],
                               args["v_cache"], args["out"], args.get("lse"), stream=0)

    assert pf([10], [33]) == cp.E_INVALID                 # c > C
    assert pf([-1], [3]) == cp.E_INVALID                  # L < 0
    assert pf([120], [9]) == cp.E_INVALID                 # L + c > P*S
    assert pf([1], [1], q=0) == cp.E_INVALID              # NULL
    assert pf([1], [1], out=A + 2) == cp.E_INVALID        # misaligned
    assert pf([1], [1], lse=A + 4) == cp.E_INVALID        # misaligned lse
    assert pf([], []) == cp.E_INVALID                     # no sequences
    assert pf([0] * 129, [1] * 129) == cp.E_UNSUPPORTED   # too many sequences
    assert pf([5], [0]) == cp.OK                          # nothing to do: no launch
    assert ctx.write_kv_raw([10], [33], A, A, A, A, stream=0) == cp.E_INVALID
    assert ctx.write_kv_raw([0], [0], A, A, A, A, stream=0) == cp.OK
    big = cp.Context(8, 2, 128, 1, 1 << 20, 1 << 20)
    n = 2100 * 128
    assert big.prefill_raw([0], [n], A, A, A, A, A, A, stream=0) in (cp.E_INVALID, cp.E_UNSUPPORTED)


def _filled_rows(L, P, S):
    fill = oracle.shard_fill(L, P)
    return {s * S + j for s in range(P) for j in range(int(fill[s]))}


WALK_CASES = [(0, 2, 8), (1, 1, 1), (5, 3, 2), (127, 1, 200), (128, 1, 128), (129, 2, 100),
              (1000, 8, 130), (777, 8, 8013), (60001, 8, 8013), (3000, 8, 8013), (300, 4, 75),
              (50, 7, 9)] + [(w.cache_lens[0], w.shards, w.shard_capacity) for w in ALL]


@pytest.mark.parametrize("L,P,S", WALK_CASES)
def test_cache_walk_covers_filled_rows_once(lib, L, P, S):
    ctx = cp.Context(2, 1, 128, P, S, 16)
    tiles, masks = ctx.cache_walk(L)
    assert np.all(np.diff(tiles) > 0), "tiles visited in increasing order, each once"
    seen = set()
    for t, m in zip(tiles, masks):
        bits = [(int(m[c // 32]) >> (c % 32)) & 1 for c in range(128)]
        assert any(bits), "a visited tile has at least one valid column"
        seen |= {t * 128 + c for c in range(128) if bits[c]}
    assert seen == _filled_rows(L, P, S)


def test_cache_walk_tile_count_is_minimal_for_aligned_shards(lib):
    # 32k shape: 8 shards of 3584 filled rows, 128-aligned: 224 full tiles.
    ctx = cp.Context(32, 2, 256, 8, 4096, 4096)
    tiles, masks = ctx.cache_walk(28672)
    assert len(tiles) == 224 and np.all(masks == 0xFFFFFFFF)


# ---------------------------------------------------------------- split-KV
@pytest.mark.parametrize("L,P,S", [(1000, 4, 300), (5000, 8, 700), (777, 8, 100), (129, 2, 65),
                                   (40000, 8, 5003), (3, 8, 1)])
def test_cache_walk_from_equals_the_tail_of_the_walk(lib, L, P, S):
    """A split-KV piece starting at virtual tile `first` skips whole shard
    ranges; it must visit exactly the rest of the full walk, same masks."""
    ctx = cp.Context(2, 1, 128, P, S, 16)
    tiles, masks = ctx.cache_walk(L)
    for first in sorted({0, 1, 2, len(tiles) // 3, len(tiles) // 2, len(tiles) - 1, len(tiles),
                         len(tiles) + 5}):
        t2, m2 = ctx.cache_walk(L, first)
        assert np.array_equal(t2, tiles[first:]), first
        assert np.array_equal(m2, masks[first:]), first


def _expected_split(ctx, cache_lens, chunk_lens, nq, hd, t):
    """Pieces and workspace of a forced split at most t tiles long, from the
    cache walk's tile counts: a walk of n > t tiles becomes ceil(n / t) pieces,
    each writing the block's valid rows."""
    blocks, rows = 0, 0
    for L, c in zip(cache_lens, chunk_lens):
        nc = len(ctx.cache_walk(L)[0])
        for qb in range(-(-c // 128)):
            n = nc + qb + 1
            k = -(-n // t) if n > t else 1
            blocks += k
            if k > 1:
                rows += k * min(128, c - 128 * qb)
    a256 = lambda x: (x + 255) // 256 * 256
    ws = a256(rows * nq * hd * 4) + a256(rows * nq * 4) if rows else 0
    return ws, blocks


@pytest.mark.parametrize("t", [1, 3, 16, 1000])
def test_splitkv_forced_plan_sizes(lib, t):
    ctx = cp.Context(8, 2, 128, 4, 4000, 384)
    cl, ch = [0, 1000, 129, 12000], [300, 1, 384, 77]
    ws, blocks = ctx.splitkv_workspace(cl, ch, t)
    assert (ws, blocks) == _expected_split(ctx, cl, ch, 8, 128, t)


def test_splitkv_automatic_policy(lib):
    """Automatic: a prefill-sized batch is never split; a decode step against
    a long cache is cut into about one piece per SM's share."""
    ctx = cp.Context(32, 2, 256, 8, 16400, 4096)
    ws, blocks = ctx.splitkv_workspace([126976], [4096], 0)
    assert ws == 0 and blocks == 32
    ws, blocks = ctx.splitkv_workspace([126976], [1], 0)
    assert ws > 0 and 1 < blocks <= 64
    # Pieces of a decode row hold 1 row x NQ heads x (HD + 1) floats each.
    a256 = lambda x: (x + 255) // 256 * 256
    assert ws == a256(blocks * 32 * 256 * 4) + a256(blocks * 32 * 4)


def test_splitkv_registration_checks(lib):
    ctx = cp.Context(8, 2, 128, 2, 64, 32)
    with pytest.raises(cp.CpattnError) as e:
        ctx.set_splitkv(None, -1)
    assert e.value.status == cp.E_INVALID
    st = ctx.lib.cpattn_set_splitkv(ctx._h, 256 + 16, 1 << 20, 0)  # not 256-byte aligned
    assert st == cp.E_INVALID
    assert ctx.lib.cpattn_set_splitkv(ctx._h, 4096, 1 << 20, 0) == cp.OK
    assert ctx.lib.cpattn_set_splitkv(ctx._h, None, 0, 0) == cp.OK  # off again


def test_splitkv_workspace_too_small_is_refused_before_launch(lib):
    ctx = cp.Context(8, 2, 128, 4, 4000, 64)
    cl, ch = [12000], [5]
    need, _ = ctx.splitkv_workspace(cl, ch, 4)
    assert need > 0
    assert ctx.lib.cpattn_set_splitkv(ctx._h, 4096, need - 256, 4) == cp.OK
    A = 256
    st = ctx.prefill_raw(cl, ch, A, A, A, A, A, A, None, stream=0)
    assert st == cp.E_INVALID and "split-KV workspace" in ctx.last_error()


def test_v_staging_registration_checks(lib):
    """Staging applies to an fp16 V cache only, and wants 16-byte alignment."""
    bf = cp.Context(8, 2, 128, 2, 64, 32)
    assert bf.lib.cpattn_set_v_staging(bf._h, 4096, 1 << 20) == cp.E_INVALID
    assert "fp16 V cache only" in bf.last_error()
    assert bf.lib.cpattn_set_v_staging(bf._h, None, 0) == cp.OK  # off is always fine
    f16 = cp.Context(8, 2, 128, 2, 64, 32, v_cache_f16=True)
    assert f16.lib.cpattn_set_v_staging(f16._h, 4096 + 8, 1 << 20) == cp.E_INVALID
    assert f16.lib.cpattn_set_v_staging(f16._h, 4096, 1 << 20) == cp.OK
    assert f16.lib.cpattn_set_v_staging(f16._h, None, 0) == cp.OK


@pytest.mark.parametrize("num_seqs", [1, 3, 128])
def test_v_staging_bytes(lib, num_seqs):
    ctx = cp.Context(32, 4, 128, 8, 8013, 4096, v_cache_f16=True)
    assert ctx.v_staging_bytes(num_seqs) == num_seqs * 4096 * 4 * 128 * 2
    for bad in (0, 129):
        with pytest.raises(cp.CpattnError) as e:
            ctx.v_staging_bytes(bad)
        assert e.value.status == cp.E_INVALID


def test_v_staging_too_small_is_refused_before_launch(lib):
    ctx = cp.Context(8, 2, 128, 4, 4000, 64, v_cache_f16=True)
    need = ctx.v_staging_bytes(2)
    assert ctx.lib.cpattn_set_v_staging(ctx._h, 4096, need - 16) == cp.OK
    A = 256
    st = ctx.prefill_raw([100, 7], [64, 5], A, A, A, A, A, A, None, stream=0)
    assert st == cp.E_INVALID and "V staging buffer" in ctx.last_error()
    # Enough for one sequence, not for two.
    assert ctx.lib.cpattn_set_v_staging(ctx._h, 4096, ctx.v_staging_bytes(1)) == cp.OK
    st = ctx.prefill_raw([100, 7], [64, 5], A, A, A, A, A, A, None, stream=0)
    assert st == cp.E_INVALID and "V staging buffer" in ctx.last_error()
    # The fused-write and two-launch entry points stage too, and refuse alike.
    st = ctx.prefill_write_kv_raw([100, 7], [64, 5], A, A, A, A, A, A, None, stream=0)
    assert st == cp.E_INVALID and "V staging buffer" in ctx.last_error()
    cl, ch = (ctypes.c_int32 * 2)(100, 7), (ctypes.c_int32 * 2)(64, 5)
    ws = ctypes.c_uint64()
    assert ctx.lib.cpattn_two_launch_workspace(ctx._h, 2, ctypes.byref(ws)) == cp.OK
    st = ctx.lib.cpattn_prefill_two_launch(ctx._h, 2, cl, ch, A, A, A, A, A, A, None, 4096,
                                           ws.value, None)
    assert st == cp.E_INVALID and "V staging buffer" in ctx.last_error()


def test_pingpong_plans_per_sm(lib):
    """Two query tiles per CTA: every SM is an executor of head pairs, so a
    short chunk against a long cache is cut into more pieces than for CTA
    pairs (one executor per two SMs); at HD = 256 the mode runs as 2-SM
    pairs and plans exactly like them."""
    plans = {}
    for mode in ("mma2", "pingpong"):
        for hd in (128, 256):
            ctx = cp.Context(8, 2, hd, 8, 8000, 128, pairing=mode)
            plans[mode, hd] = ctx.splitkv_workspace([60000], [100], 0)
            ctx.close()
    assert plans["pingpong", 256] == plans["mma2", 256]
    assert plans["pingpong", 128][1] > plans["mma2", 128][1] > 1
