"""Pins of the CPU oracle against things other than itself.

Each ``pin_*`` raises AssertionError when the oracle disagrees with a brute
force, a closed form, a library routine, a hand-worked example or an
invariant.  ``test_oracle_pins.py`` runs them as tests;
``test_oracle_mutations.py`` plants mistakes in the oracle and checks that
some pin fails for each one.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from oracle import attention as oatt
from helpers import golden, make_case
from workloads import generate, small

TOL = 1e-12


def _valid(w):
    """Boolean [T] mask of valid chunk rows."""
    m = np.zeros(w.tokens, dtype=bool)
    for b, c in enumerate(w.chunk_lens):
        m[b * w.chunk: b * w.chunk + c] = True
    return m


def _close(a, b, tol=TOL, what=""):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    assert np.all(np.isfinite(a)) and np.all(np.isfinite(b)), f"{what}: non-finite values"
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"{what}: max |diff| {err:.3e} > {tol:.1e}"


SMALL_CASES = [
    small("a", (5,), (4,), 6, nq=4, nkv=2, hd=8, shards=2, seed=11),
    small("b", (0, 3), (3, 1), 4, nq=4, nkv=2, hd=8, shards=3, seed=12),
    small("c", (7,), (1,), 1, nq=2, nkv=2, hd=8, shards=1, seed=13),
    small("d", (11, 0, 2), (5, 6, 0), 6, nq=2, nkv=1, hd=4, shards=4, seed=14),
    small("e", (9,), (7,), 8, nq=6, nkv=3, hd=8, shards=2, seed=15, peaky_frac=0.2),
]


def pin_layout_golden():
    g = golden("striped_layout.json")
    P = g["P"]
    s, j = oracle.shard_of_token(np.array(g["tokens"]), P)
    assert list(s) == g["shard"] and list(j) == g["row"], "stripe mapping"
    for key, fill in g["fill"].items():
        L = int(key.split("=")[1])
        assert list(oracle.shard_fill(L, P)) == fill, f"shard fill {key}"
    # logical -> striped -> logical round trip on a ragged length
    rng = np.random.default_rng(0)
    rows = rng.integers(0, 65535, size=(10, 2, 4), dtype=np.uint16)
    cache = oracle.build_striped_cache([rows], 2, P, 4, 4, fill=7)
    for t in range(10):
        assert np.array_equal(cache[0, :, g["shard"][t], g["row"][t], :], rows[t]), f"token {t}"
    assert np.array_equal(oracle.read_logical(cache, 0, 10), rows)


def pin_write_kv():
    g = golden("striped_layout.json")["write_case"]
    P, S, L, c, C = 3, g["S"], g["L"], g["c"], g["C"]
    rng = np.random.default_rng(1)
    NKV, HD = 2, 4
    k_new = rng.integers(0, 0x7F00, size=(C, NKV, HD), dtype=np.uint16)
    v_new = rng.integers(0, 0x7F00, size=(C, NKV, HD), dtype=np.uint16)
    kc = np.full((1, NKV, P, S, HD), 0x7F7F, dtype=np.uint16)
    vc = kc.copy()
    oracle.write_kv_ref(kc, vc, k_new, v_new, [L], [c], C)
    expect_k = np.full_like(kc, 0x7F7F)
    expect_v = expect_k.copy()
    for i, (s, j) in enumerate(g["dest"]):
        expect_k[0, :, s, j, :] = k_new[i]
        expect_v[0, :, s, j, :] = v_new[i]
    assert np.array_equal(kc, expect_k) and np.array_equal(vc, expect_v), "write_kv golden"
    # multi-sequence: every written row is the source row, the rest untouched
    w = small("wkv", (0, 5, 17), (4, 0, 6), 6, nq=2, nkv=2, hd=4, shards=4, shard_capacity=6)
    kn = rng.integers(0, 0x7F00, size=(w.tokens, 2, 4), dtype=np.uint16)
    kc = np.full((3, 2, 4, 6, 4), 0x7F7F, dtype=np.uint16)
    oracle.write_kv_ref(kc, kc.copy(), kn, kn, w.cache_lens, w.chunk_lens, w.chunk)
    written = 0
    for b in range(3):
        for i in range(w.chunk_lens[b]):
            t = w.cache_lens[b] + i
            assert np.array_equal(kc[b, :, t % 4, t // 4, :], kn[b * 6 + i]), (b, i)
            written += 1
    assert int(np.sum(np.any(kc != 0x7F7F, axis=-1))) == written * 2, "rows touched"


def pin_worked_example():
    g = golden("worked_softmax.json")
    ln2 = math.log(2.0)
    q = np.array(g["q_ln2_units"], dtype=np.float64)[:, None, :] * ln2
    kc = np.array(g["k_cache"], dtype=np.float64)[:, None, :]
    vc = np.array(g["v_cache"], dtype=np.float64)[:, None, :]
    kn = np.array(g["k_new"], dtype=np.float64)[:, None, :]
    vn = np.array(g["v_new"], dtype=np.float64)[:, None, :]
    L, c, C = g["cache_len"], g["chunk_len"], g["chunk"]
    for P in (1, 2):
        S = (L + C + P - 1) // P
        kcs = oracle.build_striped_cache([kc], 1, P, S, 2, fill=0.0, dtype=np.float64)
        vcs = oracle.build_striped_cache([vc], 1, P, S, 2, fill=0.0, dtype=np.float64)
        for scale, qs in ((1.0, q), (0.5, 2 * q)):
            o, lse = oracle.attend_ref(qs, kn, vn, kcs, vcs, [L], [c], C, scale)
            expect = np.array(g["out_num"], dtype=np.float64) / np.array(g["out_den"])[:, None]
            _close(o[:, 0, :], expect, 1e-14, "worked example O")
            _close(lse[:, 0], np.log(g["lse_of"]), 1e-14, "worked example LSE")
            o2, l2 = oracle.attend_rows_ref(qs, kn, vn, kcs, vcs, [L], [c], C, scale,
                                            [(0, 0), (1, 0)])
            _close(o2, expect, 1e-14, "worked example rows")
            _close(l2, np.log(g["lse_of"]), 1e-14, "worked example rows LSE")


def pin_brute_force():
    for w in SMALL_CASES:
        case = make_case(w)
        inp = case.inputs
        bo, bl = oracle.brute_force_ref(inp.q, inp.k_cache, inp.v_cache, inp.k_new, inp.v_new,
                                        w.cache_lens, w.chunk_lens, w.chunk, w.scale)
        o, l = case.oracle_full()
        v = _valid(w)
        _close(o[v], bo[v], TOL, f"{w.name}: O vs brute force")
        _close(l[v], bl[v], TOL, f"{w.name}: LSE vs brute force")
        samples = [(t, h) for t in np.nonzero(v)[0] for h in range(w.num_q_heads)]
        ro, rl = case.oracle_rows(samples)
        _close(ro, np.stack([bo[t, h] for t, h in samples]), TOL, f"{w.name}: rows vs brute")
        _close(rl, np.array([bl[t, h] for t, h in samples]), TOL, f"{w.name}: rows LSE")


def pin_lse_merge():
    """Cache-only and current-only softmaxes merged by LSE equal the fused one
    (the two-launch variant the PR removed computes the same thing)."""
    for w in SMALL_CASES[:4]:
        case = make_case(w)
        args = (case.f64("q"), case.f64("k_new"), case.f64("v_new"), case.f64("k_cache"),
                case.f64("v_cache"), w.cache_lens, w.chunk_lens, w.chunk, w.scale)
        o, l = oracle.attend_ref(*args)
        o1, l1 = oracle.attend_region_ref(*args, region="cache")
        o2, l2 = oracle.attend_region_ref(*args, region="current")
        mo, ml = oracle.lse_merge(o1, l1, o2, l2)
        v = _valid(w)
        _close(mo[v], o[v], TOL, f"{w.name}: merged O")
        _close(ml[v], l[v], TOL, f"{w.name}: merged LSE")


def pin_row_sums():
    for w in SMALL_CASES[:3]:
        case = make_case(w)
        for b, (L, c) in enumerate(zip(w.cache_lens, w.chunk_lens)):
            if c == 0:
                continue
            for h in range(w.num_q_heads):
                p = oracle.attention_probs_ref(case.f64("q"), case.f64("k_new"),
                                               case.f64("v_new"), case.f64("k_cache"),
                                               case.f64("v_cache"), w.cache_lens, w.chunk_lens,
                                               w.chunk, w.scale, b, h)
                _close(p.sum(axis=1), np.ones(c), TOL, "row sums")
                cur = p[:, L:]
                upper = np.triu(np.ones((c, c), dtype=bool), k=1)
                assert np.all(cur[upper] == 0.0), "future chunk keys must get zero weight"
                assert np.all(p[:, :L] > 0) and np.all(cur[~upper] > 0), "visible keys weigh > 0"


def pin_equal_keys():
    """All keys equal => O_i is the plain mean of the visible values."""
    w = small("eq", (6, 0, 13), (5, 4, 3), 5, nq=4, nkv=2, hd=8, shards=3, seed=21)
    inp = generate(w)
    rng = np.random.default_rng(3)
    kvec = rng.standard_normal((w.num_kv_heads, w.head_dim))
    kcl = [np.broadcast_to(kvec, x.shape).copy() for x in inp.k_cache]
    kn = np.broadcast_to(kvec, inp.k_new.shape).copy()
    vcl = [x.float().numpy().astype(np.float64) for x in inp.v_cache]
    vn = inp.v_new.float().numpy().astype(np.float64)
    S = w.shard_capacity
    kcs = oracle.build_striped_cache(kcl, w.num_kv_heads, w.shards, S, w.head_dim, 0.0, np.float64)
    vcs = oracle.build_striped_cache(vcl, w.num_kv_heads, w.shards, S, w.head_dim, 0.0, np.float64)
    o, _ = oracle.attend_ref(inp.q, kn, vn, kcs, vcs, w.cache_lens, w.chunk_lens, w.chunk, w.scale)
    G = w.group
    for b, (L, c) in enumerate(zip(w.cache_lens, w.chunk_lens)):
        for h in range(w.num_q_heads):
            g = h // G
            csum = vcl[b][:, g].sum(axis=0) if L else np.zeros(w.head_dim)
            for i in range(c):
                chunk_sum = vn[b * w.chunk: b * w.chunk + i + 1, g].sum(axis=0)
                expect = (csum + chunk_sum) / (L + i + 1)
                _close(o[b * w.chunk + i, h], expect, 1e-13, f"equal keys b={b} h={h} i={i}")


def _sdpa(q, k, v, mask, scale):
    """torch SDPA in float64: q [n, HD], k/v [m, HD], mask [n, m] bool or None."""
    qt, kt, vt = (torch.from_numpy(np.ascontiguousarray(x))[None, None] for x in (q, k, v))
    m = None if mask is None else torch.from_numpy(mask)[None, None]
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m,
                                                            scale=scale)[0, 0].numpy()


def pin_sdpa():
    # L = 0: plain causal self-attention; GQA by repeating kv heads.
    w = small("sd0", (0,), (9,), 9, nq=4, nkv=2, hd=16, shards=2, seed=31)
    case = make_case(w)
    o, _ = case.oracle_full()
    q, kn, vn = case.f64("q"), case.f64("k_new"), case.f64("v_new")
    for h in range(4):
        g = h // 2
        qt = torch.from_numpy(q[:, h])[None, None]
        kt = torch.from_numpy(np.ascontiguousarray(kn[:, g]))[None, None]
        vt = torch.from_numpy(np.ascontiguousarray(vn[:, g]))[None, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True,
                                                               scale=w.scale)[0, 0].numpy()
        _close(o[:, h], ref, 1e-13, "SDPA causal, L=0")
    # c = 1: one query over all L cached keys plus itself, no mask at all.
    w = small("sd1", (13,), (1,), 1, nq=2, nkv=1, hd=16, shards=3, seed=32)
    case = make_case(w)
    o, _ = case.oracle_full()
    inp = case.inputs
    k_all = np.concatenate([inp.k_cache[0][:, 0].double().numpy(), case.f64("k_new")[:1, 0]])
    v_all = np.concatenate([inp.v_cache[0][:, 0].double().numpy(), case.f64("v_new")[:1, 0]])
    for h in range(2):
        ref = _sdpa(case.f64("q")[:1, h], k_all, v_all, None, w.scale)
        _close(o[:1, h], ref, 1e-13, "SDPA single query")
    # general: explicit boolean mask over [cache | chunk]
    w = small("sd2", (10,), (6,), 6, nq=2, nkv=2, hd=16, shards=4, seed=33)
    case = make_case(w)
    o, _ = case.oracle_full()
    inp = case.inputs
    mask = np.zeros((6, 16), dtype=bool)
    for i in range(6):
        mask[i, :10] = True
        mask[i, 10:10 + i + 1] = True
    for h in range(2):
        k_all = np.concatenate([inp.k_cache[0][:, h].double().numpy(), case.f64("k_new")[:, h]])
        v_all = np.concatenate([inp.v_cache[0][:, h].double().numpy(), case.f64("v_new")[:, h]])
        ref = _sdpa(case.f64("q")[:, h], k_all, v_all, mask, w.scale)
        _close(o[:, h], ref, 1e-13, "SDPA masked")


def pin_layout_invariance():
    """The shard count and capacity are addressing only: results are identical."""
    base = small("li", (23, 4), (5, 7), 7, nq=4, nkv=2, hd=8, shards=1, seed=41)
    ref = None
    for P, pad in ((1, 0), (2, 3), (3, 0), (8, 5)):
        w = base.with_(shards=P, shard_capacity=(30 + P - 1) // P + pad)
        o, l = make_case(w).oracle_full()
        if ref is None:
            ref = (o, l)
            continue
        v = _valid(w)
        assert np.array_equal(o[v], ref[0][v]) and np.array_equal(l[v], ref[1][v]), f"P={P}"


def pin_single_key():
    """Row 0 of a sequence with an empty cache sees exactly one key: O = V_0."""
    w = small("sk", (0,), (3,), 3, nq=2, nkv=1, hd=8, shards=2, seed=51)
    case = make_case(w)
    o, l = case.oracle_full()
    q, kn, vn = case.f64("q"), case.f64("k_new"), case.f64("v_new")
    for h in range(2):
        assert np.array_equal(o[0, h], vn[0, 0]), "single key returns its value exactly"
        _close(l[0, h], w.scale * math.fsum(q[0, h] * kn[0, 0]), 1e-14, "single key LSE")


def pin_large_logits():
    """Logits near 1e4: max subtraction keeps it finite; the largest key wins."""
    HD = 4
    q = np.array([[[1.0, 0, 0, 0]]])                                     # [1, 1, HD]
    kc = np.array([[[10.0, 0, 0, 0]], [[20.0, 0, 0, 0]], [[5.0, 0, 0, 0]]])
    vc = np.arange(3 * HD, dtype=np.float64).reshape(3, 1, HD)
    kn = np.array([[[12.0, 0, 0, 0]]])
    vn = np.full((1, 1, HD), -1.0)
    kcs = oracle.build_striped_cache([kc], 1, 2, 2, HD, 0.0, np.float64)
    vcs = oracle.build_striped_cache([vc], 1, 2, 2, HD, 0.0, np.float64)
    o, l = oracle.attend_ref(q, kn, vn, kcs, vcs, [3], [1], 1, 1000.0)
    _close(o[0, 0], vc[1, 0], 1e-12, "hard max picks the largest key")
    _close(l[0, 0], 20000.0, 1e-9, "LSE of a hard max")


def pin_f16_conversion():
    """bf16 -> binary16 (IEEE 754 conversion to a narrower format, round to
    nearest even) over every bf16 pattern, against an integer restatement:
    values in binary16's normal range keep their value exactly; below 2^-14
    the result is the nearest multiple of 2^-24 (ties to even, Python's
    round); from 65520 up it is infinite."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    x = oracle.bits_to_f64(bits)
    h = oracle.bf16_to_f16_bits(bits)
    y = oracle.f16_bits_to_f64(h)
    fin = np.isfinite(x)
    ax = np.abs(x)
    normal = fin & (ax >= 2.0 ** -14) & (ax <= 65504.0)
    assert np.array_equal(y[normal], x[normal]), "normal range is exact"
    sub = fin & (ax < 2.0 ** -14)
    for xi, hi in zip(x[sub], h[sub]):
        n = round(abs(float(xi)) * 2.0 ** 24)       # ties to even
        sign = 0x8000 if math.copysign(1.0, float(xi)) < 0 else 0
        assert int(hi) == (sign | n), (xi, hex(int(hi)))
    big = fin & (ax >= 65520.0)
    assert np.all(np.isinf(y[big])) and np.array_equal(np.sign(y[big]), np.sign(x[big]))
    # binary16 decode at fixed patterns
    fixed = {0x3C00: 1.0, 0xC000: -2.0, 0x7BFF: 65504.0, 0x0001: 2.0 ** -24, 0x0400: 2.0 ** -14,
             0x3555: 0.333251953125, 0xFC00: -math.inf}
    for b, v in fixed.items():
        assert oracle.f16_bits_to_f64(np.array([b], dtype=np.uint16))[0] == v, hex(b)


def pin_write_kv_f16():
    """An fp16 V cache receives each written V value converted; K and the
    untouched rows are as in the bf16 write."""
    w = small("wkv16", (0, 5, 17), (4, 0, 6), 6, nq=2, nkv=2, hd=4, shards=4, shard_capacity=6)
    rng = np.random.default_rng(3)
    kn = rng.integers(0, 0x7F00, size=(w.tokens, 2, 4), dtype=np.uint16)
    vn = rng.integers(0, 0x4700, size=(w.tokens, 2, 4), dtype=np.uint16)  # |v| < 2^15
    kc = np.full((3, 2, 4, 6, 4), 0x1234, dtype=np.uint16)
    vc = kc.copy()
    kc2, vc2 = kc.copy(), vc.copy()
    oracle.write_kv_ref(kc, vc, kn, vn, w.cache_lens, w.chunk_lens, w.chunk, v_f16=True)
    oracle.write_kv_ref(kc2, vc2, kn, vn, w.cache_lens, w.chunk_lens, w.chunk)
    assert np.array_equal(kc, kc2), "K is written as in the bf16 cache"
    for b in range(3):
        for i in range(w.chunk_lens[b]):
            t = w.cache_lens[b] + i
            got = oracle.f16_bits_to_f64(vc[b, :, t % 4, t // 4, :])
            want = oracle.bits_to_f64(vn[b * 6 + i])
            small_ = np.abs(want) < 2.0 ** -14
            assert np.array_equal(got[~small_], want[~small_]), (b, i)
            assert np.all(np.abs(got[small_] - want[small_]) <= 2.0 ** -25), (b, i)
    assert np.array_equal(vc == 0x1234, vc2 == 0x1234), "the same rows are written"
