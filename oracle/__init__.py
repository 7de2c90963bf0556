"""CPU oracle for chunked-prefill GQA attention -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct float64 restatement of what the fused
prefill computes, written from the TPU PR "PCP: in-kernel ring cache phase,
fused with the current phase" (Summary and Design sections) and the striped
KV-cache write that PR's Testing section checks bit-exact.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA path never calls it, and it never
calls the CUDA path: the two share no code.  Inputs come from the seeded
generators in ``workloads`` (random draws only).

Parity status: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (brute force, closed forms, library special
cases, invariants) and ``tests/test_oracle_mutations.py`` (planted mistakes
that the pins must catch).
"""
from .striped import (bf16_bits, bf16_to_f16_bits, bits_to_f64, build_striped_cache,
                      f16_bits_to_f64, read_logical, shard_fill, shard_of_token, write_kv_ref)
from .attention import (attend_ref, attend_region_ref, attend_rows_ref, attention_probs_ref,
                        brute_force_ref, kv_head_of, lse_merge)

__all__ = ["bf16_bits", "bf16_to_f16_bits", "f16_bits_to_f64", "bits_to_f64", "build_striped_cache", "read_logical", "shard_fill",
           "shard_of_token", "write_kv_ref", "attend_ref", "attend_rows_ref",
           "attend_region_ref", "attention_probs_ref", "brute_force_ref", "kv_head_of", "lse_merge"]
