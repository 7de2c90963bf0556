"""Chunked-prefill GQA attention -- float64 oracle (test infrastructure).

What the fused prefill computes, restated from the TPU PR "PCP: in-kernel
ring cache phase, fused with the current phase":

* Summary: the cache rounds and the causal current phase are walked with ONE
  shared online softmax -- so the result is a single softmax over the union
  of the two key sets, not two softmaxes merged afterwards.
* Design: the current region is causal; the cache region is masked only by
  its length (every cached token is visible to every chunk row); pad rows of
  a chunk shorter than C are discarded by the caller.

Hence, for sequence b, query head h (kv head g = h div G) and valid chunk row
i < c_b, with L = L_b:

    keys   K = [cache tokens 0..L-1]  ++  [chunk tokens 0..i]
    s_k    = scale * <q_i, k_k>
    O_i    = sum_k softmax(s)_k v_k,     LSE_i = log sum_k exp(s_k)

computed in float64 with max subtraction, in logical token order (the order
of a softmax sum does not change it; the striped layout is only addressing).
The cache is read through the oracle's own inverse of the striped layout.

Readings of points the pages leave open (each checked by a pin):
  causal diagonal inclusive (key i visible to row i); cache fully visible;
  q head h uses kv head h div G; no positional terms inside attention; pad
  rows are NaN here (unspecified).
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from typing import Iterable, Sequence

import numpy as np

from . import striped

ROW_BLOCK = 256


def kv_head_of(h: int, group: int) -> int:
    """GQA map: q head h reads kv head h div G (contiguous groups)."""
    return h // group


def visible_mask(L: int, rows: np.ndarray, n_cur: int) -> np.ndarray:
    """[len(rows), L + n_cur] bool: all L cache keys, and chunk keys j <= i."""
    rows = np.asarray(rows)
    cur = np.arange(n_cur)[None, :] <= rows[:, None]
    return np.concatenate([np.ones((rows.size, L), dtype=bool), cur], axis=1)


def logits_of(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """s[i, k] = scale * <q_i, k_k>."""
    return scale * (q @ k.T)


def softmax_rows(logits: np.ndarray, mask: np.ndarray):
    """Masked softmax over the last axis (fp64, max subtracted) -> (probs, lse)."""
    s = np.where(mask, logits, -np.inf)
    m = s.max(axis=1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe)
    tot = e.sum(axis=1, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        probs = e / tot
        lse = (m_safe + np.log(tot))[:, 0]
    return probs, lse


def as_f64(x) -> np.ndarray:
    """float64 view of an input: torch tensors are converted, and uint16 arrays
    are taken as bf16 bit patterns and decoded exactly."""
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().float().numpy()
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return striped.bits_to_f64(x)
    return x.astype(np.float64, copy=False)


def _keys(k_cache, v_cache, k_new, v_new, b: int, g: int, L: int, c: int, chunk: int):
    """Visible-key candidates of (b, g) in logical order: cache then chunk."""
    kc = striped.read_logical(k_cache, b, L)[:, g, :]
    vc = striped.read_logical(v_cache, b, L)[:, g, :]
    kn = k_new[b * chunk: b * chunk + c, g, :]
    vn = v_new[b * chunk: b * chunk + c, g, :]
    return np.concatenate([kc, kn], axis=0), np.concatenate([vc, vn], axis=0)


def _head_job(args):
    (q, k_all, v_all, L, c, scale, rows_sel) = args
    rows = np.arange(c) if rows_sel is None else np.asarray(rows_sel)
    out = np.empty((rows.size, q.shape[-1]))
    lse = np.empty(rows.size)
    for r0 in range(0, rows.size, ROW_BLOCK):
        rr = rows[r0: r0 + ROW_BLOCK]
        logits = logits_of(q[rr], k_all, scale)
        probs, l = softmax_rows(logits, visible_mask(L, rr, c))
        out[r0: r0 + rr.size] = probs @ v_all
        lse[r0: r0 + rr.size] = l
    return out, lse


def attend_ref(q, k_new, v_new, k_cache, v_cache, cache_lens: Sequence[int],
               chunk_lens: Sequence[int], chunk: int, scale: float, threads: int = 1):
    """Full fused-prefill result.

    q [B*C, NQ, HD]; k_new, v_new [B*C, NKV, HD]; k_cache, v_cache striped
    [B, NKV, P, S, HD] (float arrays or torch tensors).  Returns
    (O [B*C, NQ, HD] float64 with NaN pad rows, LSE [B*C, NQ] float64 natural
    log, NaN pad rows).
    """
    q, k_new, v_new = as_f64(q), as_f64(k_new), as_f64(v_new)
    k_cache, v_cache = as_f64(k_cache), as_f64(v_cache)
    T, NQ, HD = q.shape
    NKV = k_new.shape[1]
    G = NQ // NKV
    out = np.full((T, NQ, HD), np.nan)
    lse = np.full((T, NQ), np.nan)
    jobs, where = [], []
    for b, (L, c) in enumerate(zip(cache_lens, chunk_lens)):
        if c == 0:
            continue
        for h in range(NQ):
            g = kv_head_of(h, G)
            k_all, v_all = _keys(k_cache, v_cache, k_new, v_new, b, g, L, c, chunk)
            jobs.append((q[b * chunk: b * chunk + c, h, :], k_all, v_all, L, c, scale, None))
            where.append((b, h, c))
    if threads > 1:
        with ThreadPoolExecutor(threads) as ex:
            results = list(ex.map(_head_job, jobs))
    else:
        results = [_head_job(j) for j in jobs]
    for (b, h, c), (o, l) in zip(where, results):
        out[b * chunk: b * chunk + c, h, :] = o
        lse[b * chunk: b * chunk + c, h] = l
    return out, lse


def attend_rows_ref(q, k_new, v_new, k_cache, v_cache, cache_lens, chunk_lens, chunk: int,
                    scale: float, samples: Iterable[tuple]):
    """Oracle for individual (token, q head) outputs, for sampling at full size.

    ``samples`` are (token index in [0, B*C), q head) naming a valid row.
    Inputs may be float arrays or uint16 bf16 bit patterns; only the rows
    needed are decoded, so full-size caches stay compact.
    Returns (O [n, HD], LSE [n]) float64.
    """
    NQ = q.shape[1]
    NKV = k_new.shape[1]
    G = NQ // NKV
    outs, lses = [], []
    keys = {}
    for tok, h in samples:
        b, i = divmod(int(tok), chunk)
        L, c = int(cache_lens[b]), int(chunk_lens[b])
        if i >= c:
            raise ValueError(f"token {tok} is a pad row (row {i} >= chunk length {c})")
        g = kv_head_of(int(h), G)
        if (b, g) not in keys:
            kc = as_f64(striped.read_logical(np.asarray(k_cache), b, L)[:, g, :])
            vc = as_f64(striped.read_logical(np.asarray(v_cache), b, L)[:, g, :])
            kn = as_f64(k_new[b * chunk: b * chunk + c, g, :])
            vn = as_f64(v_new[b * chunk: b * chunk + c, g, :])
            keys[(b, g)] = (np.concatenate([kc, kn]), np.concatenate([vc, vn]))
        k_all, v_all = keys[(b, g)]
        qi = as_f64(q[b * chunk: b * chunk + i + 1, int(h), :])
        o, l = _head_job((qi, k_all, v_all, L, c, scale, [i]))
        outs.append(o[0])
        lses.append(l[0])
    return np.stack(outs), np.array(lses)


def attention_probs_ref(q, k_new, v_new, k_cache, v_cache, cache_lens, chunk_lens, chunk: int,
                        scale: float, b: int, h: int):
    """The probability matrix [c_b, L_b + c_b] of one (sequence, q head)."""
    q, k_new, v_new = as_f64(q), as_f64(k_new), as_f64(v_new)
    k_cache, v_cache = as_f64(k_cache), as_f64(v_cache)
    NQ, NKV = q.shape[1], k_new.shape[1]
    L, c = int(cache_lens[b]), int(chunk_lens[b])
    g = kv_head_of(h, NQ // NKV)
    k_all, _ = _keys(k_cache, v_cache, k_new, v_new, b, g, L, c, chunk)
    logits = logits_of(q[b * chunk: b * chunk + c, h, :], k_all, scale)
    probs, _ = softmax_rows(logits, visible_mask(L, np.arange(c), c))
    return probs


def attend_region_ref(q, k_new, v_new, k_cache, v_cache, cache_lens, chunk_lens, chunk: int,
                      scale: float, region: str):
    """One region alone -- the removed two-launch variant's partial results.

    region "cache": every valid row over the L_b cached keys only;
    region "current": every valid row over chunk keys 0..i only.
    Returns (O, LSE) like :func:`attend_ref`; a row with no keys in the region
    has O = 0 and LSE = -inf.
    """
    q, k_new, v_new = as_f64(q), as_f64(k_new), as_f64(v_new)
    k_cache, v_cache = as_f64(k_cache), as_f64(v_cache)
    T, NQ, HD = q.shape
    NKV = k_new.shape[1]
    G = NQ // NKV
    out = np.full((T, NQ, HD), np.nan)
    lse = np.full((T, NQ), np.nan)
    for b, (L, c) in enumerate(zip(cache_lens, chunk_lens)):
        for h in range(NQ):
            g = kv_head_of(h, G)
            k_all, v_all = _keys(k_cache, v_cache, k_new, v_new, b, g, L, c, chunk)
            mask = visible_mask(L, np.arange(c), c)
            if region == "cache":
                mask[:, L:] = False
            elif region == "current":
                mask[:, :L] = False
            else:
                raise ValueError(region)
            logits = logits_of(q[b * chunk: b * chunk + c, h, :], k_all, scale)
            probs, l = softmax_rows(logits, mask)
            out[b * chunk: b * chunk + c, h] = np.nan_to_num(probs, nan=0.0) @ v_all
            lse[b * chunk: b * chunk + c, h] = l
    return out, lse


def lse_merge(o1, lse1, o2, lse2):
    """Combine two partial softmax results over disjoint key sets.

    With weights w_r = exp(LSE_r - max): O = (w1 O1 + w2 O2) / (w1 + w2),
    LSE = max + log(w1 + w2).  This is the merge the PR's two-launch variant
    needed and the fused kernel avoids.
    """
    m = np.maximum(lse1, lse2)
    w1 = np.exp(lse1 - m)
    w2 = np.exp(lse2 - m)
    tot = w1 + w2
    o = (w1[..., None] * o1 + w2[..., None] * o2) / tot[..., None]
    return o, m + np.log(tot)


def brute_force_ref(q, k_cache_logical, v_cache_logical, k_new, v_new, cache_lens, chunk_lens,
                    chunk: int, scale: float):
    """Scalar triple loop over the LOGICAL inputs (tiny shapes only).

    Enumerates every (row, key) pair one by one with Python floats and
    math.fsum -- no arrays, no striped layout, none of the helpers above.
    """
    q, k_new, v_new = as_f64(q), as_f64(k_new), as_f64(v_new)
    kcl = [as_f64(x) for x in k_cache_logical]
    vcl = [as_f64(x) for x in v_cache_logical]
    T, NQ, HD = q.shape
    NKV = k_new.shape[1]
    G = NQ // NKV
    out = np.full((T, NQ, HD), np.nan)
    lse = np.full((T, NQ), np.nan)
    for b in range(len(cache_lens)):
        L, c = cache_lens[b], chunk_lens[b]
        for h in range(NQ):
            g = h // G
            for i in range(c):
                qi = q[b * chunk + i, h]
                keys, vals = [], []
                for t in range(L):
                    keys.append(kcl[b][t, g])
                    vals.append(vcl[b][t, g])
                for j in range(i + 1):
                    keys.append(k_new[b * chunk + j, g])
                    vals.append(v_new[b * chunk + j, g])
                logits = [scale * math.fsum(float(qi[d]) * float(k[d]) for d in range(HD))
                          for k in keys]
                mx = max(logits)
                ws = [math.exp(s - mx) for s in logits]
                tot = math.fsum(ws)
                for d in range(HD):
                    out[b * chunk + i, h, d] = math.fsum(w * float(v[d]) for w, v in zip(ws, vals)) / tot
                lse[b * chunk + i, h] = mx + math.log(tot)
    return out, lse
