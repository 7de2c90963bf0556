"""Benchmark: one prefill step of chunked-prefill GQA attention on GB300.

A step is the whole hot path over one chunk: the strided KV-cache write of
the chunk (cpattn_write_kv) and the fused cache+current prefill
(cpattn_prefill).  The default workload is the 32k-context shape (cache
28672 + chunk 4096, NQ=32, NKV=2, HD=256, 8 striped shards, 1% of keys
doubled), seeded synthetic bf16 N(0,1) data.

    python bench.py [--steps K] [--warmup W] [--config 32k] [--gpus N]
    python bench.py --impl reference      # the CPU oracle on a bounded sample

Prints ONE JSON line (rank 0).  Under torchrun each rank runs an
independent replica of the workload (no data-path collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from workloads import BY_NAME, Workload, generate  # noqa: E402

PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20


def load_peaks():
    try:
        with open(PEAKS_PATH) as f:
            return json.load(f), "measured"
    except OSError:
        return FALLBACK_PEAKS, "fallback"


# Device sources each profiled kernel is built from, and the work plan that
# shapes its launch; a DRAM record holds while these are unchanged.
KERNEL_SOURCES = {
    "prefill": ("prefill.cuh", "prefill_pair.cuh", "prefill_pingpong.cuh", "walk.cuh", "ptx.cuh",
                "plan.h"),
    "write_kv": ("write_kv.cuh",),
}


def csrc_hash(kernel: str) -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "long_context_chunked_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def prefill_kernel_name(w, pairing: str = "mma2") -> str:
    """The prefill kernel the library launches for this workload: paired heads
    (cpattn_config.pairing, default 2-SM MMA) when the group size is even."""
    mode = os.environ.get("CPATTN_PAIRING", pairing) if w.group % 2 == 0 else "none"
    if mode == "pingpong" and w.head_dim == 128:
        return "prefill_kernel_pingpong<128>"
    if mode in ("mma2", "pingpong"):
        return "prefill_kernel_pair2<%d>" % w.head_dim
    return "prefill_kernel<%d>" % w.head_dim


def profiled_traffic(kernel: str, key: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current sources of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(key)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("csrc_hash") != csrc_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.first = 0

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            # nvidia-smi takes a while to start: wait for its first sample so
            # that a short timed region is sampled from its start; samples
            # taken before the region are not counted.
            t0 = time.time()
            while not self.lines and time.time() - t0 < 3.0 and self.proc.poll() is None:
                time.sleep(0.01)
        except OSError:
            self.proc = None
        self.first = len(self.lines)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.06)  # one more sample interval: the region's tail
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines[self.first:]:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ device
class DeviceState:
    """Device-resident inputs of one workload: Q and the chunk's K/V in token
    order, and the striped caches filled with the logical prefix by the
    library's own KV write."""

    def __init__(self, w: Workload, device, fast_p: bool = False, variant: str = "fused",
                 v_f16: bool = False, pairing: str = "mma2"):
        import torch
        import long_context_chunked_gb300 as cp
        self.w = w
        self.variant = variant
        inp = generate(w)
        self.inp = inp
        self.ctx = cp.Context.for_workload(w, fast_p=fast_p, v_cache_f16=v_f16, pairing=pairing)
        stage_v(self.ctx, w.num_seqs, device)
        self.q = inp.q.to(device)
        self.k_new = inp.k_new.to(device)
        self.v_new = inp.v_new.to(device)
        shape = (w.num_seqs, w.num_kv_heads, w.shards, w.shard_capacity, w.head_dim)
        self.k_cache = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        self.v_cache = torch.zeros(shape, dtype=torch.float16 if v_f16 else torch.bfloat16,
                                   device=device)
        self.out = torch.zeros_like(self.q)
        self.workspace = None
        if variant == "two_launch":
            self.workspace = torch.empty(self.ctx.two_launch_workspace(w.num_seqs),
                                         dtype=torch.uint8, device=device)
        lmax = max(w.cache_lens)
        if lmax:
            fill = cp.Context(w.num_q_heads, w.num_kv_heads, w.head_dim, w.shards,
                              w.shard_capacity, lmax, w.scale, v_cache_f16=v_f16)
            kl = torch.zeros((w.num_seqs * lmax, w.num_kv_heads, w.head_dim), dtype=torch.bfloat16)
            vl = torch.zeros_like(kl)
            for b, L in enumerate(w.cache_lens):
                kl[b * lmax: b * lmax + L] = inp.k_cache[b]
                vl[b * lmax: b * lmax + L] = inp.v_cache[b]
            fill.write_kv([0] * w.num_seqs, list(w.cache_lens), kl.to(device), vl.to(device),
                          self.k_cache, self.v_cache)
            fill.close()
        torch.cuda.synchronize()

    def write_kv(self, stream=None):
        w = self.w
        if self.variant == "fused_write":  # the write happens inside prefill()
            return
        self.ctx.write_kv(w.cache_lens, w.chunk_lens, self.k_new, self.v_new, self.k_cache,
                          self.v_cache, stream)

    def prefill(self, stream=None):
        w = self.w
        if self.variant == "two_launch":
            self.ctx.prefill_two_launch(w.cache_lens, w.chunk_lens, self.q, self.k_new,
                                        self.v_new, self.k_cache, self.v_cache, self.out,
                                        self.workspace, None, stream)
            return
        if self.variant == "fused_write":
            self.ctx.prefill_write_kv(w.cache_lens, w.chunk_lens, self.q, self.k_new,
                                      self.v_new, self.k_cache, self.v_cache, self.out, None,
                                      stream)
            return
        self.ctx.prefill(w.cache_lens, w.chunk_lens, self.q, self.k_new, self.v_new,
                         self.k_cache, self.v_cache, self.out, None, stream)


def time_steps(st: DeviceState, steps: int, warmup: int, flush):
    """Per-step device times (ms) of write_kv + prefill, and of prefill alone,
    with an L2 flush between steps (outside the timed events); flush=None
    times them back to back with L2 left warm."""
    import torch
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        st.write_kv()
        st.prefill()
    if st.ctx.sync_status() != 0:
        raise RuntimeError("device status after warm-up: " + st.ctx.last_error())
    step_ms, prefill_ms = [], []
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1, e2 in ev:
        if flush is not None:
            flush.zero_()
        e0.record(stream)
        st.write_kv()
        e1.record(stream)
        st.prefill()
        e2.record(stream)
    torch.cuda.synchronize()
    for e0, e1, e2 in ev:
        step_ms.append(e0.elapsed_time(e2))
        prefill_ms.append(e1.elapsed_time(e2))
    if st.ctx.sync_status() != 0:
        raise RuntimeError("device status after timing: " + st.ctx.last_error())
    return step_ms, prefill_ms


def max_abs_valid(st: DeviceState) -> float:
    """max |O| over the valid output rows of the last step (it bounds the
    oracle's max |O_ref| within the parity bar; the parity tests report
    max |O_ref| itself)."""
    w = st.w
    rows = [st.out[b * w.chunk: b * w.chunk + c] for b, c in enumerate(w.chunk_lens) if c]
    return max(float(r.abs().max().item()) for r in rows)


def measure_config(w: Workload, device, flush, steps: int, warmup: int, v_f16: bool,
                   peak: float, fast_p: bool = False) -> dict:
    """One workload's step (write_kv + prefill), timed as the headline is:
    L2 flushed between steps, CUDA events on the launching stream, SM clocks
    sampled during the timed region."""
    import torch
    st = DeviceState(w, device, fast_p=fast_p, v_f16=v_f16)
    torch.cuda.synchronize()
    with ClockSampler(device.index or 0) as clk:
        step_ms, prefill_ms = time_steps(st, steps, warmup, flush)
    flops = w.attention_flops()
    pf, ms = statistics.mean(prefill_ms), statistics.mean(step_ms)
    rec = {"workload": w.name, "description": w.description, "steps": steps,
           "v_cache": "f16" if v_f16 else "bf16", "precision": precision_label(fast_p, v_f16),
           "ms": round(ms, 4), "prefill_ms": round(pf, 4),
           "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
           "prefill_tflops": round(flops / (pf * 1e-3) / 1e12, 2),
           "frac": round(flops / (pf * 1e-3) / 1e12 / peak, 4),
           "kernel": prefill_kernel_name(w), "max_abs_out": round(max_abs_valid(st), 4),
           "clocks": clk.summary()}
    del st
    torch.cuda.empty_cache()
    return rec


def same_run_peaks(device) -> dict:
    """The roofline denominators re-measured in this run, on this GPU: a bf16
    8192^3 torch.matmul (cuBLAS; best of 10, CUDA events) and a 2 GiB device
    copy (read + write bytes, best of 10), with SM clocks sampled meanwhile."""
    import torch
    n = 8192
    a = torch.randn(n, n, device=device, dtype=torch.bfloat16)
    b = torch.randn(n, n, device=device, dtype=torch.bfloat16)
    src = torch.empty(1 << 30, dtype=torch.bfloat16, device=device).fill_(1.0)
    dst = torch.empty_like(src)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    with ClockSampler(device.index or 0) as clk:
        for _ in range(3):
            a @ b
        mm = []
        for _ in range(10):
            e0, e1 = ev(), ev()
            e0.record()
            a @ b
            e1.record()
            torch.cuda.synchronize()
            mm.append(e0.elapsed_time(e1))
        cp_ms = []
        for _ in range(10):
            e0, e1 = ev(), ev()
            e0.record()
            dst.copy_(src)
            e1.record()
            torch.cuda.synchronize()
            cp_ms.append(e0.elapsed_time(e1))
    res = {"bf16_tflops": round(2 * n ** 3 / (min(mm) * 1e-3) / 1e12, 1),
           "hbm_gbs": round(2 * src.numel() * 2 / (min(cp_ms) * 1e-3) / 1e9, 1),
           "how": "torch.matmul bf16 8192^3 and a 2 GiB copy_, best of 10 each, in this run",
           "clocks": clk.summary()}
    del a, b, src, dst
    torch.cuda.empty_cache()
    return res


def time_e2e(st: DeviceState, steps: int, warmup: int, slots: int = 2):
    """The step through the public API with inputs in pinned host memory: the
    host->device copy of Q, K_new, V_new, write_kv + prefill, and the
    device->host copy of O, every step.  Uploads, kernels and downloads run on
    three streams into double-buffered device tensors, so step i+1's upload
    and step i-1's download overlap step i's kernels, as a serving loop would
    run them."""
    import torch
    w = st.w
    hq = st.inp.q.pin_memory()
    hk = st.inp.k_new.pin_memory()
    hv = st.inp.v_new.pin_memory()
    ho = [torch.empty_like(hq).pin_memory() for _ in range(slots)]
    dev = st.q.device
    bufs = [dict(q=torch.empty_like(st.q), k=torch.empty_like(st.k_new),
                 v=torch.empty_like(st.v_new), o=torch.empty_like(st.out)) for _ in range(slots)]
    # Non-default streams: the legacy default stream would serialise them.
    up = torch.cuda.Stream(device=dev)  # host -> device
    ks = torch.cuda.Stream(device=dev)  # kernels
    dn = torch.cuda.Stream(device=dev)  # device -> host
    ev = lambda: torch.cuda.Event()
    kernels_done = [ev() for _ in range(slots)]  # the slot's last kernels finished
    output_free = [ev() for _ in range(slots)]   # the slot's last output downloaded
    for stream in (up, ks, dn):
        stream.wait_stream(torch.cuda.current_stream(device=dev))
    for e in kernels_done + output_free:
        e.record(ks)

    def one(i):
        s = i % slots
        b = bufs[s]
        with torch.cuda.stream(up):
            up.wait_event(kernels_done[s])
            b["q"].copy_(hq, non_blocking=True)
            b["k"].copy_(hk, non_blocking=True)
            b["v"].copy_(hv, non_blocking=True)
            uploaded = ev()
            uploaded.record(up)
        ks.wait_event(uploaded)
        ks.wait_event(output_free[s])
        if st.variant != "fused_write":
            st.ctx.write_kv(w.cache_lens, w.chunk_lens, b["k"], b["v"], st.k_cache, st.v_cache,
                            ks)
        if st.variant == "fused_write":
            st.ctx.prefill_write_kv(w.cache_lens, w.chunk_lens, b["q"], b["k"], b["v"],
                                    st.k_cache, st.v_cache, b["o"], None, ks)
        elif st.variant == "two_launch":
            st.ctx.prefill_two_launch(w.cache_lens, w.chunk_lens, b["q"], b["k"], b["v"],
                                      st.k_cache, st.v_cache, b["o"], st.workspace, None, ks)
        else:
            st.ctx.prefill(w.cache_lens, w.chunk_lens, b["q"], b["k"], b["v"], st.k_cache,
                           st.v_cache, b["o"], None, ks)
        kernels_done[s].record(ks)
        with torch.cuda.stream(dn):
            dn.wait_event(kernels_done[s])
            ho[s].copy_(b["o"], non_blocking=True)
            output_free[s].record(dn)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(up)
    for i in range(steps):
        one(i)
    ks.wait_stream(up)
    ks.wait_stream(dn)
    e1.record(ks)
    torch.cuda.synchronize(dev)
    if st.ctx.sync_status() != 0:
        raise RuntimeError("device status after e2e: " + st.ctx.last_error())
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho[0].numel() * ho[0].element_size()
    return e0.elapsed_time(e1) / steps, h2d, d2h


# ------------------------------------------------------------- CPU oracle
def cpu_sample(w: Workload, budget_rows: int = 384, heads: int = 2):
    """Time the fp64 oracle, as it stands, on a bounded slice of the workload:
    the first sequence, `heads` q heads of kv head 0, the first `budget_rows`
    chunk rows, the full cache.  Returns (TFLOP/s, seconds, description)."""
    import oracle
    inp = generate(w)
    L = w.cache_lens[0]
    rows = min(budget_rows, w.chunk_lens[0])
    hd = w.head_dim
    q = inp.q[:w.chunk, :heads]
    kn = inp.k_new[:w.chunk, :1]
    vn = inp.v_new[:w.chunk, :1]
    kc = oracle.build_striped_cache([oracle.bf16_bits(inp.k_cache[0][:, :1])], 1, w.shards,
                                    w.shard_capacity, hd, 0)
    vc = oracle.build_striped_cache([oracle.bf16_bits(inp.v_cache[0][:, :1])], 1, w.shards,
                                    w.shard_capacity, hd, 0)
    kcf, vcf = oracle.bits_to_f64(kc), oracle.bits_to_f64(vc)
    threads = min(heads, os.cpu_count() or 1)
    t0 = time.perf_counter()
    oracle.attend_ref(q, kn, vn, kcf, vcf, [L], [rows], w.chunk, w.scale, threads=threads)
    dt = time.perf_counter() - t0
    flops = 4 * hd * heads * (rows * L + rows * (rows + 1) // 2)
    desc = (f"{w.name}: sequence 0, {heads} q heads of kv head 0, chunk rows 0..{rows - 1}, "
            f"full cache of {L} tokens ({flops / 1e9:.1f} GFLOP), {threads} worker threads "
            f"(one per q head) on a host of {os.cpu_count()} cores")
    return flops / dt / 1e12, dt, desc, threads


# ------------------------------------------------------------------- main
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate_max(value: float, device=None) -> float:
    """Max of a per-rank timing over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm: rank 0 only, bounded samples."""
    if rank != 0:
        return
    w = BY_NAME[args.config]
    # One worker thread per q head, as many heads of kv head 0 as the host
    # has cores (the oracle's BLAS calls may use more threads inside).
    heads = max(1, min(os.cpu_count() or 1, w.group))
    vals = []
    for _ in range(args.warmup):
        cpu_sample(w, budget_rows=args.ref_rows, heads=heads)
    for _ in range(args.steps):
        tf, dt, desc, threads = cpu_sample(w, budget_rows=args.ref_rows, heads=heads)
        vals.append((tf, dt))
    v = statistics.median(t for t, _ in vals)
    sec = statistics.median(d for _, d in vals)
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) bf16 inputs)",
        "config": {"workload": w.name, "description": w.description},
        "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores,
                         "threads": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


METRIC = "fused prefill attention TFLOP/s per chunk (write_kv + prefill) on 1 GB300"

# The pages' per-request cumulative prefill TTFT (TPU v7x-8, pcp=8, CH=4k,
# NQ=32, NKV=2, HD=256, bf16), fused ring variant -- context only.
PAGES_TTFT_MS = {8192: 2.55, 16384: 6.29, 32768: 17.23, 65536: 53.05, 131072: 180.6,
                 262144: 661.0, 1048576: 9769.0}


def run_cumulative(contexts, fast_p=False, seed=7, v_f16=False, emit=True):
    """Every 4096-token chunk of one request of each context length, back to
    back on one stream: write the chunk into the striped cache, then prefill it
    against everything before it.  Returns one record per context (and prints
    each as a JSON line when emit)."""
    import torch
    import long_context_chunked_gb300 as cp
    dev = torch.device("cuda", 0)
    C, NQ, NKV, HD, P = 4096, 32, 2, 256, 8
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(C, NQ, HD, generator=gen).to(torch.bfloat16).to(dev)
    kn = torch.randn(C, NKV, HD, generator=gen).to(torch.bfloat16).to(dev)
    vn = torch.randn(C, NKV, HD, generator=gen).to(torch.bfloat16).to(dev)
    out = torch.empty_like(q)
    records = []
    for n in contexts:
        S = (n + P - 1) // P
        kc = torch.zeros((1, NKV, P, S, HD), dtype=torch.bfloat16, device=dev)
        vc = torch.zeros_like(kc, dtype=torch.float16 if v_f16 else torch.bfloat16)
        ctx = cp.Context(NQ, NKV, HD, P, S, C, 0.0, fast_p, v_f16)
        stage_v(ctx, 1, dev)
        chunks = n // C

        def request():
            for k in range(chunks):
                ctx.write_kv([k * C], [C], kn, vn, kc, vc)
                ctx.prefill([k * C], [C], q, kn, vn, kc, vc, out)

        request()  # warm-up (also fills the cache)
        torch.cuda.synchronize()
        # Several requests back to back (one for the longest): a single
        # request after an idle GPU runs at boost clocks the next does not.
        reps = 5 if n <= 131072 else 1
        times = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            request()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        if ctx.sync_status() != 0:
            raise RuntimeError(ctx.last_error())
        ms = statistics.median(times)
        flops = sum(4 * HD * NQ * (C * k * C + C * (C + 1) // 2) for k in range(chunks))
        rec = {"mode": "cumulative_prefill", "context": n, "chunks": chunks,
               "request_ms": round(ms, 3), "request_ms_min": round(min(times), 3),
               "requests_timed": reps, "tflops": round(flops / ms / 1e9, 1),
               "precision": precision_label(fast_p, v_f16),
               "v_cache": "f16" if v_f16 else "bf16",
               "pages_tpu_v7x8_fused_ring_ms": PAGES_TTFT_MS.get(n)}
        records.append(rec)
        if emit:
            print(json.dumps(rec), flush=True)
        del kc, vc, ctx
    return records


# Small-chunk and decode workloads for split-KV (NQ=32, NKV=2, HD=256, P=8,
# the pages' model shape): (name, cache lengths, chunk lengths).
SPLITKV_CASES = [
    ("decode_1x128k", [126976], [1]),
    ("decode_8x32k", [32768] * 8, [1] * 8),
    ("chunk37_15k", [15000], [37]),
    ("chunk128_4x64k", [65536] * 4, [128] * 4),
]


def run_splitkv(fast_p=False, reps=20, seed=11, v_f16=False):
    """Each small-chunk workload fused (one launch) and split-KV (automatic
    plan: pieces + merge; the same single launch when the plan cuts nothing),
    alternating rep by rep, L2 flushed before every rep, CUDA events on the
    launching stream.  Prints one JSON line per workload with both times, the
    plan's work blocks, and the split time against the HBM roofline of its
    algorithmic bytes (the K/V prefix read once, Q, O)."""
    import torch
    import long_context_chunked_gb300 as cp
    dev = torch.device("cuda", 0)
    NQ, NKV, HD, P = 32, 2, 256, 8
    peaks, peak_kind = load_peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    gen = torch.Generator().manual_seed(seed)
    for name, cl, ch in SPLITKV_CASES:
        B, C = len(cl), max(max(ch), 1)
        S = (max(l + c for l, c in zip(cl, ch)) + P - 1) // P
        q = torch.randn(B * C, NQ, HD, generator=gen).to(torch.bfloat16).to(dev)
        kn = torch.randn(B * C, NKV, HD, generator=gen).to(torch.bfloat16).to(dev)
        vn = torch.randn(B * C, NKV, HD, generator=gen).to(torch.bfloat16).to(dev)
        kc = torch.randn(B, NKV, P, S, HD, generator=gen).to(torch.bfloat16).to(dev)
        vc = torch.randn(B, NKV, P, S, HD, generator=gen).to(
            torch.float16 if v_f16 else torch.bfloat16).to(dev)
        out = torch.empty_like(q)
        ctx = cp.Context(NQ, NKV, HD, P, S, C, 0.0, fast_p, v_f16)
        stage_v(ctx, B, dev)
        need, blocks = ctx.splitkv_workspace(cl, ch, 0)
        ws = torch.empty(max(need // 4, 64), dtype=torch.float32, device=dev)

        def one(split):
            ctx.set_splitkv(ws if split else None, 0)
            flush.fill_(1.0)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            ctx.prefill(cl, ch, q, kn, vn, kc, vc, out)
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1)

        for _ in range(3):  # warm-up, both arms
            one(False)
            one(True)
        # The two arms alternate rep by rep, so clock or power drift during the
        # run affects both alike.
        fused, split = [], []
        for _ in range(reps):
            fused.append(one(False))
            split.append(one(True))
        if ctx.sync_status() != 0:
            raise RuntimeError(ctx.last_error())
        fused_ms, split_ms = statistics.median(fused), statistics.median(split)
        # The split step replayed from a CUDA graph: the GPU time alone, as a
        # serving loop that captures its decode step sees it (the eager arm
        # above also pays planning, tensor-map encoding and two launches on
        # the host while the GPU idles).
        ctx.set_splitkv(ws, 0)
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            ctx.prefill(cl, ch, q, kn, vn, kc, vc, out)  # warm-up on the capture stream
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph):
            ctx.prefill(cl, ch, q, kn, vn, kc, vc, out)
        gtimes = []
        for _ in range(reps):
            flush.fill_(1.0)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            graph.replay()
            e1.record()
            torch.cuda.synchronize()
            gtimes.append(e0.elapsed_time(e1))
        if ctx.sync_status() != 0:
            raise RuntimeError(ctx.last_error())
        graph_ms = statistics.median(gtimes)
        del graph
        flops = sum(4 * HD * NQ * (c * l + c * (c + 1) // 2) for l, c in zip(cl, ch))
        kv_bytes = sum(2 * NKV * HD * 2 * (l + c) for l, c in zip(cl, ch))
        io_bytes = sum(c for c in ch) * NQ * HD * 2 * 2
        gbs = (kv_bytes + io_bytes) / (graph_ms * 1e-3) / 1e9
        print(json.dumps({
            "mode": "splitkv", "workload": name, "cache_lens": cl, "chunk_lens": ch,
            "precision": precision_label(fast_p, v_f16), "v_cache": "f16" if v_f16 else "bf16",
            "row_blocks": sum(-(-c // 128) for c in ch), "work_blocks_split": blocks,
            "fused_ms": round(fused_ms, 4), "split_ms": round(split_ms, 4),
            "split_graph_ms": round(graph_ms, 4),
            "speedup": round(fused_ms / split_ms, 2),
            "split_tflops": round(flops / (graph_ms * 1e-3) / 1e12, 2),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1),
                         "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                         "frac": round(gbs / float(peaks["hbm_gbs"]), 4),
                         "peak_kind": f"HBM copy, {peak_kind}",
                         "bytes": "K/V prefix and chunk read once + Q + O",
                         "time": "split step replayed from a CUDA graph"},
            "l2": "flushed before every rep"}), flush=True)
        del q, kn, vn, kc, vc, out, ws, ctx


# fp16 V cache: stage the chunk's V in fp16 (cpattn_set_v_staging) so that
# every tile takes fp16 P with one P.V product (--v-staging off: current
# tiles keep the bf16 hi+lo pair, or fast_p).
V_STAGING = True


def stage_v(ctx, num_seqs: int, device):
    """Register a V staging buffer for batches of up to num_seqs sequences
    on an fp16-V-cache context (kept alive on the context)."""
    import torch
    if not (ctx.v_cache_f16 and V_STAGING):
        return
    n = ctx.v_staging_bytes(num_seqs)
    ctx.v_stage_buf = torch.empty(n // 2, dtype=torch.float16, device=device)
    ctx.set_v_staging(ctx.v_stage_buf)


def precision_label(fast_p: bool, v_f16: bool) -> str:
    cur = "P rounded to bf16" if fast_p else "bf16 hi+lo P pair"
    if v_f16 and V_STAGING:
        return "every tile: fp16 P x fp16 V (the chunk's V staged in fp16)"
    if v_f16:
        return f"cache tiles: fp16 P x fp16 V; current tiles: {cur}"
    return "fast_p (P rounded to bf16)" if fast_p else "accurate P (bf16 hi+lo pair)"


def traffic_key(kname: str, workload: str, fast_p: bool, v_f16: bool) -> str:
    if v_f16 and V_STAGING:  # every tile one fp16 product: fast_p does not apply
        return f"{kname}:{workload}:vf16staged"
    return f"{kname}:{workload}:{'fast_p' if fast_p else 'accurate'}" + (":vf16" if v_f16 else "")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="cpattn", choices=["cpattn", "reference"])
    ap.add_argument("--config", default="32k", choices=sorted(BY_NAME))
    ap.add_argument("--fast-p", action="store_true", help="P rounded once to bf16")
    ap.add_argument("--v-cache", default="f16", choices=["bf16", "f16"],
                    help="V cache format (default f16: cache tiles take P in fp16, one P.V "
                         "product at the accurate mode's precision; bf16: the bf16 hi+lo P "
                         "pair on every tile)")
    ap.add_argument("--v-staging", default="on", choices=["on", "off"],
                    help="fp16 V cache: stage the chunk's V in fp16 so that its tiles take "
                         "fp16 P too (default on; off: the bf16 hi+lo pair on current tiles)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--variant", default="fused", choices=["fused", "two_launch", "fused_write"],
                    help="fused_write: the KV write inside the prefill launch; "
                         "two_launch: the PR's removed variant (cache-only + current-only "
                         "launches + LSE merge), to measure what fusion saves")
    ap.add_argument("--ref-rows", type=int, default=384)
    ap.add_argument("--splitkv", action="store_true",
                    help="small-chunk and decode workloads, fused vs split-KV")
    ap.add_argument("--cumulative", default=None,
                    help="comma-separated request lengths (e.g. 8k,32k,1M): per-request "
                         "cumulative prefill instead of the step benchmark")
    ap.add_argument("--no-extras", action="store_true",
                    help="only the headline workload: skip the other configs, the bf16 V "
                         "cache record, the cumulative requests and the same-run peaks")
    args = ap.parse_args()
    global V_STAGING
    V_STAGING = args.v_staging == "on"
    world, rank, local = dist_setup()
    if args.splitkv:
        run_splitkv(fast_p=args.fast_p, v_f16=args.v_cache == "f16")
        return
    if args.cumulative:
        mult = {"k": 1024, "m": 1024 * 1024}
        ns = [int(x[:-1]) * mult[x[-1].lower()] if x[-1].lower() in mult else int(x)
              for x in args.cumulative.split(",")]
        run_cumulative(ns, fast_p=args.fast_p, v_f16=args.v_cache == "f16")
        return
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    w = BY_NAME[args.config]
    v_f16 = args.v_cache == "f16"
    st = DeviceState(w, device, fast_p=args.fast_p, variant=args.variant, v_f16=v_f16)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        step_ms, prefill_ms = time_steps(st, args.steps, args.warmup, flush)
    torch.cuda.synchronize()
    total_ms = aggregate_max(sum(step_ms), device)
    if world > 1:
        dist.barrier()
    e2e_ms, h2d, d2h = time_e2e(st, max(4, args.steps // 2), args.warmup)
    # Context beside the flushed number: the same step with L2 left warm.
    _, hot_prefill_ms = time_steps(st, min(args.steps, 20), 3, None)

    flops = w.attention_flops()
    kname = prefill_kernel_name(w)
    ms_step = total_ms / args.steps
    value = world * flops / (ms_step * 1e-3) / 1e12
    peaks, peak_kind = load_peaks()
    pf = statistics.mean(prefill_ms)
    achieved = flops / (pf * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    kv_ms = statistics.mean(s - p for s, p in zip(step_ms, prefill_ms))
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16+f16" if v_f16 else "bf16",
        "data": "synthetic (seeded N(0,1) bf16, 1% of keys doubled)",
        "config": {"workload": w.name, "description": w.description,
                   "precision": precision_label(args.fast_p, v_f16),
                   "v_cache": args.v_cache,
                   "v_staging": bool(v_f16 and V_STAGING),
                   "l2": "flushed between steps (512 MiB write)",
                   "parallelism": f"replicas x{world}", "variant": args.variant},
        "prefill_ms": round(pf, 4), "write_kv_ms": round(kv_ms, 4),
        "prefill_ms_hot_l2": round(statistics.mean(hot_prefill_ms), 4),
        "write_kv_gbs": round(w.kv_write_bytes() / (kv_ms * 1e-3) / 1e9, 1) if kv_ms > 0 else None,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "peak_kind": f"bf16 dense burst, {peak_kind}",
                     "frac_of_sustained": round(achieved / float(peaks["bf16_tflops_sustained"]), 4),
                     "kernel": kname,
                     "traffic": profiled_traffic(
                         "prefill", traffic_key(kname, w.name, args.fast_p, v_f16))},
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "note": "pinned host buffers; uploads and downloads on their own streams overlap the previous/next step's kernels"},
        # write_kv, the V staging (fp16 V cache), prefill.
        "gpu_launches": ({"fused": 2, "two_launch": 4, "fused_write": 1}[args.variant]
                         + (1 if v_f16 and V_STAGING else 0)) * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_extras and world == 1:
        # Beside the headline, every other configuration and the bf16 V cache
        # (every tile takes the bf16 hi+lo P pair, and the KV write is a pure
        # bit copy), each timed as the headline is; then whole cumulative
        # requests, and the roofline denominators re-measured in this run.
        extra_steps = max(5, min(args.steps, 20))
        per = {}
        for name in ("tiny", "8k", "128k", "varlen"):
            if name != w.name:
                per[name] = measure_config(BY_NAME[name], device, flush, extra_steps, 3,
                                           v_f16, peak, args.fast_p)
        line["per_config"] = per
        line["max_abs_out"] = round(max_abs_valid(st), 4)
        del st
        torch.cuda.empty_cache()
        line["bf16_v_cache"] = measure_config(w, device, flush, extra_steps, 3, False, peak,
                                              args.fast_p)
        line["cumulative"] = run_cumulative([8192, 32768, 131072], fast_p=args.fast_p,
                                            v_f16=v_f16, emit=False)
        sr = same_run_peaks(device)
        line["roofline"]["peak_same_run"] = sr["bf16_tflops"]
        line["roofline"]["frac_of_same_run"] = round(achieved / sr["bf16_tflops"], 4)
        line["same_run_peaks"] = sr
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # About 10 s of oracle work on a 16-core host: up to 16 q heads of kv
        # head 0 (one worker thread each) and up to 2048 chunk rows.
        tf, dt, desc, threads = cpu_sample(w, budget_rows=2048, heads=min(16, w.group))
        line["cpu_baseline"] = {"value": round(tf, 6), "unit": "TFLOP/s",
                                "cores": os.cpu_count(), "threads": threads, "kind": "oracle",
                                "sample": desc, "seconds": round(dt, 2)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
