"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins
catch every one of them -- evidence that the pins constrain the oracle rather
than restate it.  Covered: the attention arithmetic, the striped layout and
write, the LSE merge, the working precision, and the bf16 -> fp16 conversion
of the fp16 V cache."""
import numpy as np
import pytest

import oracle
import oracle_pins
from oracle import attention as oatt
from oracle import striped as ostr

PINS = sorted(n for n in dir(oracle_pins) if n.startswith("pin_"))


def _strict_causal(L, rows, n_cur):
    rows = np.asarray(rows)
    cur = np.arange(n_cur)[None, :] < rows[:, None]
    return np.concatenate([np.ones((rows.size, L), dtype=bool), cur], axis=1)


def _cache_short(L, rows, n_cur):
    rows = np.asarray(rows)
    cur = np.arange(n_cur)[None, :] <= rows[:, None]
    cache = np.ones((rows.size, L), dtype=bool)
    if L:
        cache[:, -1] = False
    return np.concatenate([cache, cur], axis=1)


def _softmax_no_max(logits, mask):
    s = np.where(mask, logits, -np.inf)
    e = np.exp(s)
    tot = e.sum(axis=1, keepdims=True)
    with np.errstate(all="ignore"):
        return e / tot, np.log(tot)[:, 0]


_orig_softmax = oatt.softmax_rows


def _lse_no_max(logits, mask):
    p, _ = _orig_softmax(logits, mask)
    s = np.where(mask, logits, -np.inf)
    m = s.max(axis=1)
    return p, np.log(np.exp(s - m[:, None]).sum(axis=1))


_orig_write = ostr.write_kv_ref


def _write_off_by_one(k_cache, v_cache, k_new, v_new, cache_lens, chunk_lens, chunk):
    return _orig_write(k_cache, v_cache, k_new, v_new, [L + 1 for L in cache_lens], chunk_lens,
                       chunk)


def _merge_swapped(o1, lse1, o2, lse2):
    m = np.maximum(lse1, lse2)
    w1, w2 = np.exp(lse1 - m), np.exp(lse2 - m)
    return (w2[..., None] * o1 + w1[..., None] * o2) / (w1 + w2)[..., None], m + np.log(w1 + w2)


_orig_as_f64 = oatt.as_f64
_orig_f16 = ostr.bf16_to_f16_bits


def _f16_toward_zero(u16):
    """bf16 -> binary16 rounded toward zero instead of to nearest even."""
    f32 = (np.asarray(u16).astype(np.uint32) << 16).view(np.float32)
    with np.errstate(over="ignore"):
        h = f32.astype(np.float16)
    hb = h.view(np.uint16).copy()
    up = np.abs(h.astype(np.float32)) > np.abs(f32)  # rounded away from zero
    hb[up] -= 1  # one step smaller in magnitude, same sign
    return hb


def _f16_flush_subnormals(u16):
    h = _orig_f16(u16).copy()
    h[(h & 0x7C00) == 0] &= 0x8000
    return h


def _f16_saturating(u16):
    h = _orig_f16(u16).copy()
    inf = (h & 0x7FFF) == 0x7C00
    h[inf] = (h[inf] & 0x8000) | 0x7BFF
    return h


def _write_v_unconverted(k_cache, v_cache, k_new, v_new, cache_lens, chunk_lens, chunk,
                         v_f16=False):
    return _orig_write(k_cache, v_cache, k_new, v_new, cache_lens, chunk_lens, chunk)

MUTANTS = {
    "gqa map h mod G": (oatt, "kv_head_of", lambda h, g: h % g),
    "causal diagonal excluded": (oatt, "visible_mask", _strict_causal),
    "last cached key hidden": (oatt, "visible_mask", _cache_short),
    "scale dropped": (oatt, "logits_of", lambda q, k, s: q @ k.T),
    "logit sign flipped": (oatt, "logits_of", lambda q, k, s: -s * (q @ k.T)),
    "no max subtraction": (oatt, "softmax_rows", _softmax_no_max),
    "LSE without max term": (oatt, "softmax_rows", _lse_no_max),
    "shard order mirrored": (ostr, "shard_of_token", lambda t, P: ((P - 1) - t % P, t // P)),
    "stripe transposed": (ostr, "shard_of_token", lambda t, P: (t // P % P, t % P + (t // P // P) * P)),
    "write lands one token late": (ostr, "write_kv_ref", _write_off_by_one),
    "merge weights swapped": (oatt, "lse_merge", _merge_swapped),
    "fp32 instead of fp64": (oatt, "as_f64", lambda x: _orig_as_f64(x).astype(np.float32).astype(np.float64)),
    "fp16 V rounded toward zero": (ostr, "bf16_to_f16_bits", _f16_toward_zero),
    "fp16 V subnormals flushed": (ostr, "bf16_to_f16_bits", _f16_flush_subnormals),
    "fp16 V overflow saturates": (ostr, "bf16_to_f16_bits", _f16_saturating),
    "fp16 V cache written unconverted": (ostr, "write_kv_ref", _write_v_unconverted),
}


def _rebind(monkeypatch, mod, name, fn):
    monkeypatch.setattr(mod, name, fn)
    # the package re-exports some names: patch those bindings too
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, fn)


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_mutant(mutant, monkeypatch):
    mod, name, fn = MUTANTS[mutant]
    _rebind(monkeypatch, mod, name, fn)
    caught = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                getattr(oracle_pins, pin)()
        except Exception as e:  # AssertionError or a crash both count as caught
            caught.append((pin, type(e).__name__))
    assert caught, f"no pin caught the planted mistake '{mutant}'"
