"""Split-KV prefill on the GPU against the fp64 oracle.

With a workspace registered, cpattn_prefill may cut a row block's tile walk
(cache tiles, then causal current tiles) into pieces on different SMs; each
piece writes fp32 O / l and its LSE for the block's valid rows, and a merge
kernel combines the pieces by LSE.  The result must meet the same bar as the
fused kernel: forced splits (pieces of 1, 2, 5 tiles: pieces that start
mid-shard, pieces of only current tiles, a diagonal tile alone) on ragged
multi-sequence cases, the automatic policy on decode-like steps, in the
paired and unpaired kernels.  The workspace sits between canary bands: no
piece may write outside the partial rows its plan gave it."""
import numpy as np
import pytest
import torch

import long_context_chunked_gb300 as cp
from gpu_helpers import DeviceCase, compare, to_f64
from helpers import make_case
from workloads import small

pytestmark = pytest.mark.gpu

WS_GUARD = 1024  # floats of canary on each side (keeps 256-byte alignment)
WS_CANARY = 0x7FBADBAD  # a NaN bit pattern no kernel writes


class Workspace:
    def __init__(self, nbytes: int):
        n = max(nbytes // 4, 1)
        self.n = n
        self.base = torch.full((WS_GUARD + n + WS_GUARD,), WS_CANARY, dtype=torch.int32,
                               device="cuda")
        self.t = self.base[WS_GUARD:WS_GUARD + n]
        assert self.t.data_ptr() % 256 == 0

    def guards_intact(self) -> bool:
        g = self.base.cpu().numpy()
        return bool(np.all(g[:WS_GUARD] == WS_CANARY) and np.all(g[WS_GUARD + self.n:] == WS_CANARY))


def _run(w, max_split_tiles, expect_split=True):
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    need, blocks = ctx.splitkv_workspace(w.cache_lens, w.chunk_lens, max_split_tiles)
    row_blocks = sum(-(-c // 128) for c in w.chunk_lens)
    if expect_split:
        assert need > 0 and blocks > row_blocks, (need, blocks, row_blocks)
    ws = Workspace(need)
    ctx.set_splitkv(ws.t, max_split_tiles)
    dc.prefill(ctx)
    ref, ref_lse = case.oracle_full()
    v = dc.valid_rows()
    out = to_f64(dc.out.bits())
    res = compare(out[v], ref[v], f"{w.name} split {max_split_tiles}")
    lse = dc.lse.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lse[v] - ref_lse[v])) < 2e-3, "LSE"
    pad = ~v
    if pad.any():
        assert np.all(dc.out.bits()[pad] == np.uint16(0x7F7F)), "pad rows written"
    assert dc.guards_intact(), "write outside an input or output buffer"
    assert ws.guards_intact(), "write outside the split-KV workspace"
    return out, res


CASES = [
    small("spA", (0, 1000, 129, 3000), (300, 1, 256, 77), 320, nq=8, nkv=2, hd=128, shards=4,
          shard_capacity=800, seed=51),
    small("spB", (5000, 1), (130, 384), 384, nq=4, nkv=1, hd=256, shards=8, seed=52),
    small("spC", (2000,), (200,), 256, nq=3, nkv=3, hd=128, shards=3, seed=53),  # unpaired
]


@pytest.mark.parametrize("t", [1, 2, 5])
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_forced_split_parity(w, t):
    _run(w, t)


@pytest.mark.parametrize("mode", ["mma2", "none", "pingpong"])
def test_forced_split_parity_pairing_modes(mode, monkeypatch):
    monkeypatch.setenv("CPATTN_PAIRING", mode)
    _run(CASES[0], 3)


DECODE = [
    small("dec256", (20000, 15000, 9000), (1, 3, 1), 64, nq=8, nkv=2, hd=256, shards=8, seed=61),
    small("dec128", (30001,), (40,), 64, nq=8, nkv=4, hd=128, shards=8, seed=62),
]


@pytest.mark.parametrize("w", DECODE, ids=[w.name for w in DECODE])
def test_automatic_split_decode(w):
    _run(w, 0)


def test_split_and_fused_agree(monkeypatch):
    """The same batch with and without splitting: both within the bar of the
    oracle, and within bf16 rounding of each other."""
    w = DECODE[0]
    split_out, _ = _run(w, 4)
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    dc.prefill(ctx)
    fused = to_f64(dc.out.bits())
    v = dc.valid_rows()
    d = np.abs(split_out[v] - fused[v])
    assert float(d.max()) <= 2e-2 and float(np.sqrt((d * d).mean())) < 2e-3


def test_workspace_off_again():
    """Registering NULL turns split-KV off: the plan then needs no workspace
    and the prefill runs fused."""
    w = DECODE[1]
    case = make_case(w)
    dc = DeviceCase(case)
    ctx = cp.Context.for_workload(w)
    need, _ = ctx.splitkv_workspace(w.cache_lens, w.chunk_lens, 2)
    ws = Workspace(need)
    ctx.set_splitkv(ws.t, 2)
    ctx.set_splitkv(None)
    dc.prefill(ctx)
    assert ws.guards_intact()
    assert np.all(ws.t.cpu().numpy() == WS_CANARY), "workspace used while split-KV was off"
    ref, _ = case.oracle_full()
    v = dc.valid_rows()
    compare(to_f64(dc.out.bits())[v], ref[v], "after turning split-KV off")


FULL_DECODE = [
    small("dec_1x128k", (126976,), (1,), 1, nq=32, nkv=2, hd=256, shards=8, seed=91),
    small("dec_8x32k", (32768,) * 8, (1,) * 8, 1, nq=32, nkv=2, hd=256, shards=8, seed=92),
]


@pytest.mark.parametrize("w", FULL_DECODE, ids=[w.name for w in FULL_DECODE])
def test_full_size_decode_every_row(w):
    """The decode workloads `bench.py --splitkv` times, at full size in the
    launch configuration it times (GQA-packed, automatic split-KV plan): a
    decode step has only NQ output rows per sequence, so every one of them
    is compared with the oracle."""
    _run(w, 0)
