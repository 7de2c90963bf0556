// LSE merge of two partial attention results over disjoint key sets -- the
// step the PCP ring-cache PR's removed two-launch variant needed after its
// cache-only and current-only launches (Summary section), kept here to
// measure what the fused kernel saves.  For each valid (token, q head) row:
//   m = max(l1, l2),  w_r = exp(l_r - m),
//   O = (w1 O1 + w2 O2) / (w1 + w2),  LSE = m + log(w1 + w2)
// A row whose sequence has no cached tokens takes the current-only part.
// HBM-bound: one thread per 8 consecutive output elements.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace cpattn {

struct MergeParams {
  const float* o1;     // [T, NQ, HD] cache-only partial (fp32)
  const float* lse1;   // [T, NQ]
  const float* o2;     // [T, NQ, HD] current-only partial
  const float* lse2;   // [T, NQ]
  __nv_bfloat16* out;  // [T, NQ, HD]
  float* lse;          // [T, NQ] or null
  int num_seqs, C, nq, hd;
  long long total;     // sum_b c_b * NQ * HD / 8 work items
  int has_cache[CPATTN_MAX_SEQS];
  long long item_prefix[CPATTN_MAX_SEQS + 1];
};

__global__ void __launch_bounds__(256) lse_merge_kernel(const __grid_constant__ MergeParams p) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const int per_row = p.hd / 8;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
       idx < p.total; idx += stride) {
    int lo = 0, hi = p.num_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.item_prefix[mid] <= idx) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const long long local = idx - p.item_prefix[b];
    const long long row = local / per_row;       // (i, h) within sequence b
    const int part = static_cast<int>(local - row * per_row);
    const long long r = static_cast<long long>(b) * p.C * p.nq + row;  // (tok * NQ + h)
    const float l2 = p.lse2[r];
    float w1 = 0.f, w2 = 1.f, lse = l2;
    if (p.has_cache[b]) {
      const float l1 = p.lse1[r];
      const float m = fmaxf(l1, l2);
      w1 = __expf(l1 - m);
      w2 = __expf(l2 - m);
      lse = m + __logf(w1 + w2);
    }
    const float inv = 1.f / (w1 + w2);
    const long long e = r * p.hd + part * 8;
    const float4 b0 = *reinterpret_cast<const float4*>(p.o2 + e);
    const float4 b1 = *reinterpret_cast<const float4*>(p.o2 + e + 4);
    float v[8] = {b0.x * w2, b0.y * w2, b0.z * w2, b0.w * w2,
                  b1.x * w2, b1.y * w2, b1.z * w2, b1.w * w2};
    if (p.has_cache[b]) {
      const float4 a0 = *reinterpret_cast<const float4*>(p.o1 + e);
      const float4 a1 = *reinterpret_cast<const float4*>(p.o1 + e + 4);
      v[0] += a0.x * w1; v[1] += a0.y * w1; v[2] += a0.z * w1; v[3] += a0.w * w1;
      v[4] += a1.x * w1; v[5] += a1.y * w1; v[6] += a1.z * w1; v[7] += a1.w * w1;
    }
    uint4 o;
    o.x = pack_bf16x2(v[0] * inv, v[1] * inv);
    o.y = pack_bf16x2(v[2] * inv, v[3] * inv);
    o.z = pack_bf16x2(v[4] * inv, v[5] * inv);
    o.w = pack_bf16x2(v[6] * inv, v[7] * inv);
    *reinterpret_cast<uint4*>(p.out + e) = o;
    if (part == 0 && p.lse != nullptr) p.lse[r] = lse;
  }
}

// Split-KV merge: a row block whose tile walk was cut into n pieces (a
// "group") has, per valid row and q head, n partial results (O_s / l_s in
// fp32 and LSE_s) over disjoint key sets; the softmax over their union is
//   m = max_s LSE_s,  w_s = exp(LSE_s - m),
//   O = sum_s w_s O_s / sum_s w_s,  LSE = m + log(sum_s w_s).
// Piece s of a group has its partial rows at part0 + s * rows.
constexpr int kMaxSplitGroups = 256;

struct SplitMergeParams {
  const float* ws_o;    // [partial rows][NQ][HD]
  const float* ws_lse;  // [partial rows][NQ]
  __nv_bfloat16* out;   // [T, NQ, HD]
  float* lse;           // [T, NQ] or null
  int num_groups, C, nq, hd;
  long long total;      // (row, head) pairs: sum over groups of rows * NQ
  int g_b[kMaxSplitGroups], g_q0[kMaxSplitGroups], g_rows[kMaxSplitGroups];
  int g_n[kMaxSplitGroups], g_part0[kMaxSplitGroups];
  long long g_prefix[kMaxSplitGroups + 1];
};

// One CTA of kMergeWarps warps per (row, head) of a group.  Every warp reads
// all n piece LSEs (a few per lane) and reduces their max and weight sum
// itself; warp w then accumulates the pieces s = w, w + kMergeWarps, ... for
// output elements 8j .. 8j + 7 in lane j, and the warps' partial sums are
// added through shared memory.  A decode step has few (row, head) pairs and
// many pieces: spreading the pieces over warps turns n dependent memory
// round trips into n / kMergeWarps.
constexpr int kMergeWarps = 8;
constexpr int kMergeMaxHd = 256;

__global__ void __launch_bounds__(32 * kMergeWarps) splitkv_merge_kernel(
    const __grid_constant__ SplitMergeParams p) {
  __shared__ float part[kMergeWarps][kMergeMaxHd];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // Launched as a programmatic dependent of the prefill kernel: the launch
  // overlaps the prefill's tail; this waits until that grid has completed
  // and its partial rows are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (long long it = blockIdx.x; it < p.total; it += gridDim.x) {
    int lo = 0, hi = p.num_groups - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.g_prefix[mid] <= it) lo = mid; else hi = mid - 1;
    }
    const int g = lo;
    const int local = static_cast<int>(it - p.g_prefix[g]);
    const int r = local / p.nq, h = local - r * p.nq;
    const int n = p.g_n[g];
    const long long pr0 = static_cast<long long>(p.g_part0[g]) + r;  // piece s: pr0 + s * rows
    const long long pstride = p.g_rows[g];
    float m = -INFINITY;
    for (int s = lane; s < n; s += 32) m = fmaxf(m, p.ws_lse[(pr0 + s * pstride) * p.nq + h]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    float wsum = 0.f;
    for (int s = lane; s < n; s += 32) wsum += __expf(p.ws_lse[(pr0 + s * pstride) * p.nq + h] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xFFFFFFFFu, wsum, o);
    const int e = lane * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (e < p.hd) {
#pragma unroll 2
      for (int s = warp; s < n; s += kMergeWarps) {
        const long long pr = pr0 + s * pstride;
        const float w = __expf(p.ws_lse[pr * p.nq + h] - m);
        const float* src = p.ws_o + (pr * p.nq + h) * p.hd + e;
        const float4 a = *reinterpret_cast<const float4*>(src);
        const float4 b = *reinterpret_cast<const float4*>(src + 4);
        acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
        acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) part[warp][e + i] = acc[i];
    }
    __syncthreads();
    // Thread t sums element t over the warps' partials.
    for (int x = threadIdx.x; x < p.hd; x += blockDim.x) {
      float v = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < kMergeWarps; ++w2) v += part[w2][x];
      part[0][x] = v;  // each element read-then-written by one thread only
    }
    __syncthreads();
    if (warp == 0 && e < p.hd) {
      const float inv = 1.f / wsum;
      const long long tok = static_cast<long long>(p.g_b[g]) * p.C + p.g_q0[g] + r;
      const float* v = &part[0][e];
      uint4 o;
      o.x = pack_bf16x2(v[0] * inv, v[1] * inv);
      o.y = pack_bf16x2(v[2] * inv, v[3] * inv);
      o.z = pack_bf16x2(v[4] * inv, v[5] * inv);
      o.w = pack_bf16x2(v[6] * inv, v[7] * inv);
      *reinterpret_cast<uint4*>(p.out + (tok * p.nq + h) * p.hd + e) = o;
      if (lane == 0 && p.lse != nullptr) p.lse[tok * p.nq + h] = m + __logf(wsum);
    }
    __syncthreads();  // part[] is reused by the next (row, head)
  }
}

}  // namespace cpattn
