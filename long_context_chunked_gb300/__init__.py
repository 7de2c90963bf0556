"""cpattn: fused chunked-prefill GQA attention on GB300 (sm_103a).

The compute path is the CUDA library ``libcpattn.so`` (C ABI, include/cpattn.h):
the striped KV-cache write and the fused cache+current prefill kernel.  This
package only loads it and marshals arguments (``binding.Context``).
"""
from .binding import (E_CUDA, E_INVALID, E_NOMEM, E_RANGE, E_TIMEOUT, E_UNSUPPORTED, EXPORTS,
                      LIB_PATH, MAX_ROW_BLOCKS, MAX_SEQS, OK, Context, CpattnError, load)

__all__ = ["Context", "CpattnError", "load", "LIB_PATH", "EXPORTS", "OK", "E_INVALID",
           "E_UNSUPPORTED", "E_CUDA", "E_NOMEM", "E_TIMEOUT", "E_RANGE", "MAX_SEQS",
           "MAX_ROW_BLOCKS"]
