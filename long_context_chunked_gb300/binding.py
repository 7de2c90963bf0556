"""ctypes binding of ``libcpattn.so`` (declared in include/cpattn.h).

Argument marshalling only: every step of the hot path runs in the CUDA
kernels of the library.  There is no fallback -- if the library is missing
or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
# CPATTN_LIBRARY overrides the library path (e.g. an instrumented build).
LIB_PATH = os.environ.get("CPATTN_LIBRARY") or os.path.join(_PKG, "libcpattn.so")

OK, E_INVALID, E_UNSUPPORTED, E_CUDA, E_NOMEM, E_TIMEOUT, E_RANGE = range(7)
MAX_SEQS = 128
MAX_ROW_BLOCKS = 2048

# Every symbol include/cpattn.h declares.
EXPORTS = ("cpattn_create", "cpattn_write_kv", "cpattn_prefill", "cpattn_sync_status",
           "cpattn_set_fault_injection", "cpattn_cache_walk", "cpattn_destroy",
           "cpattn_status_string", "cpattn_last_error", "cpattn_prefill_noalloc",
           "cpattn_two_launch_workspace", "cpattn_prefill_two_launch", "cpattn_set_splitkv",
           "cpattn_splitkv_workspace", "cpattn_cache_walk_from", "cpattn_prefill_write_kv",
           "cpattn_set_barrier_counts", "cpattn_set_v_staging", "cpattn_v_staging_bytes")

# cpattn_config.pairing values, by name.
PAIRING = {"mma2": 0, "none": 1, "pingpong": 2}
COUNT_BARS = 40      # CPATTN_COUNT_BARS
COUNT_RECORD = 200   # CPATTN_COUNT_RECORD: uint32 per CTA


class CpattnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"cpattn status {status}: {msg}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("num_shards", ctypes.c_int32),
                ("shard_capacity", ctypes.c_int32), ("chunk_size", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("fast_p", ctypes.c_int32),
                ("v_cache_f16", ctypes.c_int32), ("pairing", ctypes.c_int32),
                ("gqa_packing", ctypes.c_int32)]


_libs = {}


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load a build of the library (once per path).  Raises if it has not
    been built."""
    if path in _libs:
        return _libs[path]
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing: build it with "
                           "long_context_chunked_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I32, U32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32
    I32P = ctypes.POINTER(ctypes.c_int32)
    lib.cpattn_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(P)]
    lib.cpattn_create.restype = I32
    lib.cpattn_write_kv.argtypes = [P, I32, I32P, I32P, P, P, P, P, P]
    lib.cpattn_write_kv.restype = I32
    lib.cpattn_prefill.argtypes = [P, I32, I32P, I32P, P, P, P, P, P, P, P, P]
    lib.cpattn_prefill.restype = I32
    lib.cpattn_sync_status.argtypes = [P, P]
    lib.cpattn_sync_status.restype = I32
    lib.cpattn_set_fault_injection.argtypes = [P, I32, I32]
    lib.cpattn_set_fault_injection.restype = I32
    lib.cpattn_cache_walk.argtypes = [P, I32, I32P, ctypes.POINTER(U32), I32, I32P]
    lib.cpattn_cache_walk.restype = I32
    lib.cpattn_destroy.argtypes = [P]
    lib.cpattn_destroy.restype = None
    lib.cpattn_status_string.argtypes = [I32]
    lib.cpattn_status_string.restype = ctypes.c_char_p
    lib.cpattn_last_error.argtypes = [P]
    lib.cpattn_last_error.restype = ctypes.c_char_p
    lib.cpattn_prefill_noalloc.argtypes = [ctypes.POINTER(Config), I32, I32P, I32P] + [P] * 8
    lib.cpattn_prefill_noalloc.restype = I32
    lib.cpattn_two_launch_workspace.argtypes = [P, I32, ctypes.POINTER(ctypes.c_uint64)]
    lib.cpattn_two_launch_workspace.restype = I32
    lib.cpattn_prefill_two_launch.argtypes = [P, I32, I32P, I32P] + [P] * 8 + [ctypes.c_uint64, P]
    lib.cpattn_prefill_two_launch.restype = I32
    lib.cpattn_set_splitkv.argtypes = [P, P, ctypes.c_uint64, I32]
    lib.cpattn_set_splitkv.restype = I32
    lib.cpattn_splitkv_workspace.argtypes = [P, I32, I32P, I32P, I32,
                                             ctypes.POINTER(ctypes.c_uint64), I32P]
    lib.cpattn_splitkv_workspace.restype = I32
    lib.cpattn_cache_walk_from.argtypes = [P, I32, I32, I32P, ctypes.POINTER(U32), I32, I32P]
    lib.cpattn_cache_walk_from.restype = I32
    lib.cpattn_prefill_write_kv.argtypes = [P, I32, I32P, I32P, P, P, P, P, P, P, P, P]
    lib.cpattn_prefill_write_kv.restype = I32
    lib.cpattn_set_barrier_counts.argtypes = [P, P, ctypes.c_uint64]
    lib.cpattn_set_barrier_counts.restype = I32
    if hasattr(lib, "cpattn_set_v_staging"):  # absent from older builds (A/B timing only)
        lib.cpattn_set_v_staging.argtypes = [P, P, ctypes.c_uint64]
        lib.cpattn_set_v_staging.restype = I32
        lib.cpattn_v_staging_bytes.argtypes = [P, I32, ctypes.POINTER(ctypes.c_uint64)]
        lib.cpattn_v_staging_bytes.restype = I32
    _libs[path] = lib
    return lib


def _i32(values: Sequence[int]):
    arr = np.ascontiguousarray(np.asarray(values, dtype=np.int32))
    return arr, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _ptr(t) -> int:
    """Device pointer of a tensor, or an int passed through; None -> NULL."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Context:
    """One attention-layer shape: NQ, NKV, HD, shard count P, shard capacity S, chunk C.
    pairing: "mma2" (default), "none" or "pingpong"; gqa_packing: False turns
    the packed short-chunk form off; library: the path of another build of the
    library (e.g. the barrier-count build) to run this context on."""

    def __init__(self, num_q_heads: int, num_kv_heads: int, head_dim: int, num_shards: int,
                 shard_capacity: int, chunk_size: int, softmax_scale: float = 0.0,
                 fast_p: bool = False, v_cache_f16: bool = False, pairing: str = "mma2",
                 gqa_packing: bool = True, library: Optional[str] = None):
        self.lib = load(library or LIB_PATH)
        self.cfg = Config(num_q_heads, num_kv_heads, head_dim, num_shards, shard_capacity,
                          chunk_size, softmax_scale, int(bool(fast_p)), int(bool(v_cache_f16)),
                          PAIRING[pairing], 0 if gqa_packing else 1)
        self.v_cache_f16 = bool(v_cache_f16)
        h = ctypes.c_void_p()
        st = self.lib.cpattn_create(ctypes.byref(self.cfg), ctypes.byref(h))
        if st != OK:
            raise CpattnError(st, self.lib.cpattn_status_string(st).decode())
        self._h = h

    @classmethod
    def for_workload(cls, w, fast_p: bool = False, v_cache_f16: bool = False,
                     pairing: str = "mma2", gqa_packing: bool = True,
                     library: Optional[str] = None) -> "Context":
        return cls(w.num_q_heads, w.num_kv_heads, w.head_dim, w.shards, w.shard_capacity,
                   w.chunk, w.scale, fast_p, v_cache_f16, pairing, gqa_packing, library)

    # -- status --------------------------------------------------------
    def _check(self, st: int):
        if st != OK:
            msg = self.lib.cpattn_last_error(self._h).decode() or \
                self.lib.cpattn_status_string(st).decode()
            raise CpattnError(st, msg)

    def status(self, st: int) -> int:
        return st

    # -- entry points --------------------------------------------------
    def write_kv_raw(self, cache_lens, chunk_lens, k_new, v_new, k_cache, v_cache, stream=None) -> int:
        cl, clp = _i32(cache_lens)
        ch, chp = _i32(chunk_lens)
        return self.lib.cpattn_write_kv(self._h, len(cl), clp, chp, _ptr(k_new), _ptr(v_new),
                                        _ptr(k_cache), _ptr(v_cache), _stream(stream))

    def write_kv(self, cache_lens, chunk_lens, k_new, v_new, k_cache, v_cache, stream=None):
        self._check_tensors((k_new, v_new, k_cache), v_cache)
        self._check(self.write_kv_raw(cache_lens, chunk_lens, k_new, v_new, k_cache, v_cache,
                                      stream))

    def prefill_raw(self, cache_lens, chunk_lens, q, k_new, v_new, k_cache, v_cache, out,
                    lse=None, stream=None) -> int:
        cl, clp = _i32(cache_lens)
        ch, chp = _i32(chunk_lens)
        return self.lib.cpattn_prefill(self._h, len(cl), clp, chp, _ptr(q), _ptr(k_new),
                                       _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(out),
                                       _ptr(lse), _stream(stream))

    def prefill(self, cache_lens, chunk_lens, q, k_new, v_new, k_cache, v_cache, out, lse=None,
                stream=None):
        self._check_tensors((q, k_new, v_new, k_cache, out), v_cache)
        self._check(self.prefill_raw(cache_lens, chunk_lens, q, k_new, v_new, k_cache, v_cache,
                                     out, lse, stream))

    def prefill_write_kv_raw(self, cache_lens, chunk_lens, q, k_new, v_new, k_cache, v_cache,
                             out, lse=None, stream=None) -> int:
        cl, clp = _i32(cache_lens)
        ch, chp = _i32(chunk_lens)
        return self.lib.cpattn_prefill_write_kv(
            self._h, len(cl), clp, chp, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
            _ptr(v_cache), _ptr(out), _ptr(lse), _stream(stream))

    def prefill_write_kv(self, cache_lens, chunk_lens, q, k_new, v_new, k_cache, v_cache, out,
                         lse=None, stream=None):
        """Prefill and the chunk's KV-cache write in one launch."""
        self._check_tensors((q, k_new, v_new, k_cache, out), v_cache)
        self._check(self.prefill_write_kv_raw(cache_lens, chunk_lens, q, k_new, v_new, k_cache,
                                              v_cache, out, lse, stream))

    def two_launch_workspace(self, num_seqs: int) -> int:
        n = ctypes.c_uint64()
        self._check(self.lib.cpattn_two_launch_workspace(self._h, num_seqs, ctypes.byref(n)))
        return n.value

    def prefill_two_launch(self, cache_lens, chunk_lens, q, k_new, v_new, k_cache, v_cache, out,
                           workspace, lse=None, stream=None):
        """The removed two-launch variant (cache-only + current-only + LSE merge)."""
        self._check_tensors((q, k_new, v_new, k_cache, out), v_cache)
        cl, clp = _i32(cache_lens)
        ch, chp = _i32(chunk_lens)
        nbytes = workspace.numel() * workspace.element_size()
        self._check(self.lib.cpattn_prefill_two_launch(
            self._h, len(cl), clp, chp, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
            _ptr(v_cache), _ptr(out), _ptr(lse), _ptr(workspace), nbytes, _stream(stream)))

    def set_splitkv(self, workspace=None, max_split_tiles: int = 0):
        """Register a device workspace (a CUDA tensor, 256-byte aligned) for
        split-KV, or None to turn it off; max_split_tiles 0 = automatic."""
        nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        self._check(self.lib.cpattn_set_splitkv(self._h, _ptr(workspace), nbytes,
                                                max_split_tiles))

    def splitkv_workspace(self, cache_lens, chunk_lens, max_split_tiles: int = 0):
        """(workspace bytes, work blocks) of this batch's split-KV plan."""
        cl, clp = _i32(cache_lens)
        ch, chp = _i32(chunk_lens)
        n = ctypes.c_uint64()
        blocks = ctypes.c_int32()
        self._check(self.lib.cpattn_splitkv_workspace(self._h, len(cl), clp, chp, max_split_tiles,
                                                      ctypes.byref(n), ctypes.byref(blocks)))
        return n.value, blocks.value

    def set_v_staging(self, buffer=None):
        """fp16 V cache: register a device buffer (a CUDA tensor, 16-byte
        aligned, v_staging_bytes(num_seqs) bytes for the largest batch) in
        which the prefill calls stage the chunk's V in fp16, or None to stop
        staging."""
        nbytes = 0 if buffer is None else buffer.numel() * buffer.element_size()
        self._check(self.lib.cpattn_set_v_staging(self._h, _ptr(buffer), nbytes))

    def v_staging_bytes(self, num_seqs: int) -> int:
        """Bytes of the V staging buffer for a batch of num_seqs sequences."""
        n = ctypes.c_uint64()
        self._check(self.lib.cpattn_v_staging_bytes(self._h, num_seqs, ctypes.byref(n)))
        return n.value

    def sync_status(self, stream=None) -> int:
        """Synchronise and return the status code (E_TIMEOUT if a device wait expired)."""
        return self.lib.cpattn_sync_status(self._h, _stream(stream))

    def set_barrier_counts(self, records=None):
        """Register a zeroed device uint32 tensor of COUNT_RECORD entries per
        CTA (barrier-count build only), or None to stop counting."""
        nbytes = 0 if records is None else records.numel() * records.element_size()
        self._check(self.lib.cpattn_set_barrier_counts(self._h, _ptr(records), nbytes))

    def set_fault_injection(self, flags: int, timeout_ms: int = 0):
        self._check(self.lib.cpattn_set_fault_injection(self._h, flags, timeout_ms))

    def cache_walk(self, cache_len: int, first: int = 0):
        """(tiles int32 [n], masks uint32 [n, 4]) of the kernel's cache walk,
        from its tile `first` on (the start of a split-KV piece)."""
        n = ctypes.c_int32()
        fn = self.lib.cpattn_cache_walk_from
        self._check(fn(self._h, cache_len, first, None, None, 0, ctypes.byref(n)))
        tiles = np.zeros(max(n.value, 1), dtype=np.int32)
        masks = np.zeros((max(n.value, 1), 4), dtype=np.uint32)
        self._check(fn(self._h, cache_len, first,
                       tiles.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                       masks.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)), n.value,
                       ctypes.byref(n)))
        return tiles[:n.value], masks[:n.value]

    def last_error(self) -> str:
        return self.lib.cpattn_last_error(self._h).decode()

    def close(self):
        if getattr(self, "_h", None):
            self.lib.cpattn_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check_tensors(self, ts, v_cache):
        """bf16 tensors, and the V cache in the context's format (fp16 with
        v_cache_f16, else bf16); contiguous, on the GPU."""
        import torch
        want_v = torch.float16 if self.v_cache_f16 else torch.bfloat16
        for t, want in [(t, torch.bfloat16) for t in ts] + [(v_cache, want_v)]:
            if t is None or isinstance(t, int):
                continue
            if t.dtype != want or not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"expected a contiguous {want} CUDA tensor, got {t.dtype}")


def prefill_noalloc(cfg: Config, cache_lens, chunk_lens, q, k_new, v_new, k_cache, v_cache, out,
                    lse=None, stream=None) -> int:
    """cpattn_prefill_noalloc: the fused prefill without a context and without
    any allocation, for callers that cannot allocate device memory.  Returns
    the status code."""
    fn = load().cpattn_prefill_noalloc
    cl, clp = _i32(cache_lens)
    ch, chp = _i32(chunk_lens)
    return fn(ctypes.byref(cfg), len(cl), clp, chp, _ptr(q), _ptr(k_new), _ptr(v_new),
              _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), _stream(stream))
