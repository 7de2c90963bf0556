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

}  // namespace cpattn
