// Iteration order over one (sequence, kv head)'s striped cache.
//
// The PCP ring-cache PR (Design section) walks the cache as P ring rounds,
// one striped shard per round.  On one GPU every shard is resident, so the
// ring survives only as this order: shard 0's tiles, then shard 1's, ...
// Tiles are BKV consecutive rows of the flat shard array [P * S] of one
// (sequence, kv head), aligned to multiples of BKV -- so when S is not a
// multiple of BKV a tile straddles a shard boundary and its valid columns
// come from two shards.  A tile is visited iff it holds at least one filled
// row; a tile shared by two shards is visited once.
#pragma once

#include <cstdint>

namespace cpattn {

constexpr int kBQ = 128;   // query rows per work unit (MMA M)
constexpr int kBKV = 128;  // kv rows per tile (QK^T N, PV K)

// n_s(L): how many of the first L tokens land in shard s (stripe width one).
__host__ __device__ __forceinline__ int shard_fill(int L, int P, int s) {
  return L > s ? (L - s + P - 1) / P : 0;
}

struct CacheWalk {
  int L, P, S;
  int s;          // shard whose range is being walked (P when finished)
  int k;          // next tile index (flat rows [k*BKV, k*BKV + BKV))
  int k_last;     // last tile of shard s's range
  int prev_last;  // last tile emitted so far
  long long lo, hi;  // filled flat rows of shard s: [s*S, s*S + n_s)
  bool last_full;    // the tile returned by next() lies wholly inside [lo, hi)

  __host__ __device__ __forceinline__ void init(int L_, int P_, int S_) {
    L = L_;
    P = P_;
    S = S_;
    s = -1;
    prev_last = -1;
    next_shard();
  }

  __host__ __device__ __forceinline__ void next_shard() {
    while (true) {
      ++s;
      const int f = (s < P) ? shard_fill(L, P, s) : 0;
      if (f == 0) {  // fills are non-increasing in s: nothing further
        s = P;
        return;
      }
      const long long a = static_cast<long long>(s) * S;
      int first = static_cast<int>(a / kBKV);
      const int last = static_cast<int>((a + f - 1) / kBKV);
      if (first <= prev_last) first = prev_last + 1;
      if (first <= last) {
        k = first;
        k_last = last;
        lo = a;
        hi = a + f;
        return;
      }
    }
  }

  __host__ __device__ __forceinline__ bool done() const { return s >= P; }

  // Skip the next n tiles of the walk (a work item that starts mid-walk):
  // whole shard ranges at a time, O(P).  Skipping past the end finishes it.
  __host__ __device__ __forceinline__ void skip(int n) {
    while (n > 0 && !done()) {
      const int left = k_last - k + 1;  // tiles still to emit in shard s's range
      if (n < left) {
        k += n;
        prev_last = k - 1;
        return;
      }
      n -= left;
      prev_last = k_last;
      next_shard();
    }
  }

  // Emit the current tile index and advance.  Interior tiles of a shard's
  // range are wholly valid (last_full); only the tiles at its edges need the
  // column mask.
  __host__ __device__ __forceinline__ int next() {
    const int t = k;
    const long long r0 = static_cast<long long>(t) * kBKV;
    last_full = r0 >= lo && r0 + kBKV <= hi;
    prev_last = t;
    if (k < k_last)
      ++k;
    else
      next_shard();
    return t;
  }

  // Validity of the tile's 128 columns as four 32-bit words (bit c of word
  // c/32): column c is flat row f = tile*BKV + c, valid iff f lies within
  // the filled prefix of its shard.
  __host__ __device__ __forceinline__ void column_mask(int tile, uint32_t (&w)[4]) const {
    w[0] = w[1] = w[2] = w[3] = 0u;
    const long long r0 = static_cast<long long>(tile) * kBKV;
    const long long r1 = r0 + kBKV;
    int s0 = static_cast<int>(r0 / S);
    for (int sh = s0; sh < P && static_cast<long long>(sh) * S < r1; ++sh) {
      const long long a = static_cast<long long>(sh) * S;
      const long long b = a + shard_fill(L, P, sh);
      const long long lo = a > r0 ? a : r0;
      const long long hi = b < r1 ? b : r1;
      if (lo >= hi) continue;
      const int c0 = static_cast<int>(lo - r0), c1 = static_cast<int>(hi - r0);  // [c0, c1)
      for (int q = 0; q < 4; ++q) {
        const int qa = q * 32, qb = qa + 32;
        const int x0 = c0 > qa ? c0 : qa, x1 = c1 < qb ? c1 : qb;
        if (x0 >= x1) continue;
        const int n = x1 - x0;
        const uint32_t bits = (n == 32) ? 0xFFFFFFFFu : ((1u << n) - 1u);
        w[q] |= bits << (x0 - qa);
      }
    }
  }
};

// Number of cache tiles the walk visits for cache length L: whole shard
// ranges at a time (as skip() moves), O(P).
__host__ __device__ inline int cache_tile_count(int L, int P, int S) {
  CacheWalk w;
  w.init(L, P, S);
  int n = 0;
  while (!w.done()) {
    n += w.k_last - w.k + 1;
    w.prev_last = w.k_last;
    w.next_shard();
  }
  return n;
}

}  // namespace cpattn
