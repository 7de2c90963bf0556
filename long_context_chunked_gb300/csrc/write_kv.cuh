// Strided KV-cache write: the chunk's valid tokens, in token order, are
// copied bit for bit into their striped cache slots (PCP ring-cache PR,
// Testing section: the strided cache write must be bit-exact; the m-star
// ring_scatter op has the same pure-copy contract).
//
// HBM-bound copy.  One thread moves one 16-byte vector of K and the same
// vector of V; consecutive threads cover consecutive vectors of one source
// row, so loads and stores are fully coalesced within each HD*2-byte row.
// An fp16 V cache (v_f16) receives each V value converted from bf16 with
// round-to-nearest-even: exact for 2^-17 <= |v| <= 65504; below 2^-17 the
// value is rounded to a multiple of 2^-24 (fp16's subnormal step), so
// |v| <= 2^-25 becomes zero -- an absolute error of at most 2^-25, not
// reported.  A value beyond 65504 sets kStatusRange in *status.
#pragma once

#include <cstdint>

#include "ptx.cuh"
#include "walk.cuh"

namespace cpattn {

struct WriteKvParams {
  const uint4* k_new;
  const uint4* v_new;
  uint4* k_cache;
  uint4* v_cache;
  int* status;                            // device status word (range errors)
  int v_f16;                              // V cache in fp16
  int num_seqs, nkv, P, S, C;
  int vec_per_row;                        // HD * 2 / 16
  long long total_vecs;                   // sum_b c_b * NKV * vec_per_row
  int cache_len[CPATTN_MAX_SEQS];
  long long vec_prefix[CPATTN_MAX_SEQS + 1];  // first vector index of each sequence
};

__global__ void __launch_bounds__(256) write_kv_kernel(const __grid_constant__ WriteKvParams p) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
       idx < p.total_vecs; idx += stride) {
    // sequence of this vector: binary search in the prefix table
    int lo = 0, hi = p.num_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.vec_prefix[mid] <= idx) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const long long local = idx - p.vec_prefix[b];
    const long long row = local / p.vec_per_row;          // (i, g) row within the chunk
    const int vec = static_cast<int>(local - row * p.vec_per_row);
    const int i = static_cast<int>(row / p.nkv);
    const int g = static_cast<int>(row - static_cast<long long>(i) * p.nkv);
    const long long src = (static_cast<long long>(b) * p.C * p.nkv + row) * p.vec_per_row + vec;
    const int t = p.cache_len[b] + i;
    const long long dst_row =
        (static_cast<long long>(b * p.nkv + g) * p.P + (t % p.P)) * p.S + (t / p.P);
    const long long dst = dst_row * p.vec_per_row + vec;
    const uint4 kv = __ldg(p.k_new + src);
    uint4 vv = __ldg(p.v_new + src);
    if (p.v_f16) {
      bool overflow = false;
      vv = bf16x8_to_f16x8(vv, &overflow);
      if (overflow && p.status != nullptr) atomicCAS(p.status, kStatusOk, kStatusRange);
    }
    p.k_cache[dst] = kv;
    p.v_cache[dst] = vv;
  }
}

// The chunk's V in fp16, token order [B * C, NKV, HD] like V_new, for the
// prefill of an fp16 V cache: its current tiles then take the same fp16 P
// and single P.V product as its cache tiles.  Valid rows (token i < c_b) are
// converted as the fp16 cache write converts them (a value beyond 65504 sets
// kStatusRange); pad rows are written as zeros, so that a pad row's finite
// but out-of-range bf16 value cannot become an infinity that a masked
// (P = 0) column would turn into NaN.  HBM-bound: one 16-byte vector per
// thread, coalesced.
struct StageVParams {
  const uint4* v_new;
  uint4* v_stage;
  int* status;
  int C, nkv, vec_per_row;
  long long total_vecs;  // B * C * NKV * vec_per_row
  int chunk_len[CPATTN_MAX_SEQS];
};

__global__ void __launch_bounds__(256) stage_v_f16_kernel(const __grid_constant__ StageVParams p) {
  // The prefill kernel is launched as a programmatic dependent of this one:
  // it may start now (its blocks then occupy no SM this grid still needs,
  // since every block of this grid has started), and its producer waits for
  // this grid's completion before its first copy.
  griddep_launch_dependents();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long per_token = static_cast<long long>(p.nkv) * p.vec_per_row;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
       idx < p.total_vecs; idx += stride) {
    const long long token = idx / per_token;
    const int b = static_cast<int>(token / p.C);
    const int i = static_cast<int>(token - static_cast<long long>(b) * p.C);
    uint4 vv = make_uint4(0u, 0u, 0u, 0u);
    if (i < p.chunk_len[b]) {
      bool overflow = false;
      vv = bf16x8_to_f16x8(__ldg(p.v_new + idx), &overflow);
      if (overflow && p.status != nullptr) atomicCAS(p.status, kStatusOk, kStatusRange);
    }
    p.v_stage[idx] = vv;
  }
}

}  // namespace cpattn
