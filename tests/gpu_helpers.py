"""GPU-side test plumbing: device copies with guard bands, and the tolerance
check used by every parity test."""
from __future__ import annotations

import collections

import numpy as np
import torch

GUARD = 4096                      # int16 elements of canary before and after each buffer
CANARY = np.int16(0x7F7F)         # bf16 3.39e38, finite
MAX_ABS = 1e-2                    # max |O - O_ref| over valid rows
MAX_REL_RMS = 2e-3                # ||O - O_ref||_2 / ||O_ref||_2


class Guarded:
    """A device buffer with canary bands on both sides (bounds check without a sanitizer)."""

    def __init__(self, shape, fill_bits=None, dtype=torch.bfloat16):
        n = int(np.prod(shape))
        self.n = n
        self.shape = tuple(shape)
        self.base = torch.full((GUARD + n + GUARD,), int(CANARY), dtype=torch.int16, device="cuda")
        if fill_bits is not None:
            src = torch.from_numpy(np.ascontiguousarray(fill_bits).reshape(-1).view(np.int16))
            self.base[GUARD:GUARD + n].copy_(src.cuda())
        self.t = self.base[GUARD:GUARD + n].view(dtype).view(self.shape)

    def bits(self) -> np.ndarray:
        return self.base[GUARD:GUARD + self.n].cpu().numpy().view(np.uint16).reshape(self.shape)

    def guards_intact(self) -> bool:
        g = self.base.cpu().numpy()
        return bool(np.all(g[:GUARD] == CANARY) and np.all(g[GUARD + self.n:] == CANARY))


def to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


Parity = collections.namedtuple("Parity", "max_abs rel n_allowance max_abs_ref")


def compare(out: np.ndarray, ref: np.ndarray, what: str = "", max_abs_bar: float = None,
            rel_bar: float = None) -> Parity:
    """Parity bar against the unrounded fp64 oracle: relative RMS <= 2e-3 and
    max |diff| <= 1e-2.  Where rounding the exact value to bf16 alone moves it
    by more than half that bar (|O| >= 4, half-ulp 1.6e-2), the element may
    also differ by its own rounding error plus 5e-3: no bf16 output can do
    better there.  Returns the max |diff|, the relative RMS, how many
    elements went past the max-|diff| bar under that allowance, and
    max |O_ref|.  Below |O_ref| = 2 the allowance never exceeds the bar (a
    bf16 half-ulp there is at most 3.9e-3), which is asserted too."""
    assert out.shape == ref.shape, (out.shape, ref.shape)
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    d = out - ref
    rounding = np.abs(bf16_round(ref) - ref)
    bar_abs = MAX_ABS if max_abs_bar is None else max_abs_bar
    bar_rel = MAX_REL_RMS if rel_bar is None else rel_bar
    allowed = np.maximum(bar_abs, rounding + bar_abs / 2)
    excess = float(np.max(np.abs(d) - allowed))
    max_abs = float(np.max(np.abs(d)))
    rel = float(np.sqrt(np.sum(d * d) / np.sum(ref * ref)))
    over = np.abs(d) > bar_abs
    n_allowance = int(np.count_nonzero(over))
    assert excess <= 0 and rel <= bar_rel, \
        f"{what}: max|d|={max_abs:.3e} (<= {bar_abs} + rounding), relRMS={rel:.3e} (<= {bar_rel})"
    assert not np.any(over & (np.abs(ref) < 2)), f"{what}: allowance used where |O_ref| < 2"
    return Parity(max_abs, rel, n_allowance, float(np.max(np.abs(ref))))


class DeviceCase:
    """Device-resident inputs of a helpers.Case, with guard bands."""

    def __init__(self, case, out_fill=None):
        w = case.w
        self.case = case
        self.q = Guarded(case.q_bits.shape, case.q_bits)
        self.k_new = Guarded(case.k_new_bits.shape, case.k_new_bits)
        self.v_new = Guarded(case.v_new_bits.shape, case.v_new_bits)
        self.k_cache = Guarded(case.k_cache_bits.shape, case.k_cache_bits)
        self.v_cache = Guarded(case.v_cache_bits.shape, case.v_cache_bits,
                               dtype=torch.float16 if case.v_f16 else torch.bfloat16)
        self.out = Guarded((w.tokens, w.num_q_heads, w.head_dim))
        self.lse = torch.full((w.tokens, w.num_q_heads), float("nan"), dtype=torch.float32,
                              device="cuda")

    def prefill(self, ctx, with_lse=True):
        w = self.case.w
        ctx.prefill(w.cache_lens, w.chunk_lens, self.q.t, self.k_new.t, self.v_new.t,
                    self.k_cache.t, self.v_cache.t, self.out.t, self.lse if with_lse else None)
        st = ctx.sync_status()
        assert st == 0, f"status {st}: {ctx.last_error()}"

    def guards_intact(self) -> bool:
        return all(b.guards_intact() for b in (self.q, self.k_new, self.v_new, self.k_cache,
                                                self.v_cache, self.out))

    def valid_rows(self):
        w = self.case.w
        m = np.zeros(w.tokens, dtype=bool)
        for b, c in enumerate(w.chunk_lens):
            m[b * w.chunk: b * w.chunk + c] = True
        return m
