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
// Piece s of a group has its partial rows at part0 + s * rows.  HBM-bound:
// one thread per 8 consecutive output elements of one (row, head).
constexpr int kMaxSplitGroups = 256;

struct SplitMergeParams {
  const float* ws_o;    // [partial rows][NQ][HD]
  const float* ws_lse;  // [partial rows][NQ]
  __nv_bfloat16* out;   // [T, NQ, HD]
  float* lse;           // [T, NQ] or null
  int num_groups, C, nq, hd;
  long long total;      // sum over groups of rows * NQ * HD / 8
  int g_b[kMaxSplitGroups], g_q0[kMaxSplitGroups], g_rows[kMaxSplitGroups];
  int g_n[kMaxSplitGroups], g_part0[kMaxSplitGroups];
  long long g_prefix[kMaxSplitGroups + 1];
};

__global__ void __launch_bounds__(256) splitkv_merge_kernel(const __grid_constant__ SplitMergeParams p) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const int per_head = p.hd / 8;
  const int per_row = p.nq * per_head;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
       idx < p.total; idx += stride) {
    int lo = 0, hi = p.num_groups - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.g_prefix[mid] <= idx) lo = mid; else hi = mid - 1;
    }
    const int g = lo;
    const long long local = idx - p.g_prefix[g];
    const int r = static_cast<int>(local / per_row);         // row within the block
    const int rem = static_cast<int>(local - static_cast<long long>(r) * per_row);
    const int h = rem / per_head;
    const int part8 = rem - h * per_head;
    const int n = p.g_n[g];
    float m = -INFINITY;
    for (int s = 0; s < n; ++s) {
      const long long pr = static_cast<long long>(p.g_part0[g]) + static_cast<long long>(s) * p.g_rows[g] + r;
      m = fmaxf(m, p.ws_lse[pr * p.nq + h]);
    }
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float wsum = 0.f;
    for (int s = 0; s < n; ++s) {
      const long long pr = static_cast<long long>(p.g_part0[g]) + static_cast<long long>(s) * p.g_rows[g] + r;
      const float w = __expf(p.ws_lse[pr * p.nq + h] - m);
      wsum += w;
      const float* src = p.ws_o + (pr * p.nq + h) * p.hd + part8 * 8;
      const float4 a = *reinterpret_cast<const float4*>(src);
      const float4 b = *reinterpret_cast<const float4*>(src + 4);
      acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
      acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
    }
    const float inv = 1.f / wsum;
    const long long tok = static_cast<long long>(p.g_b[g]) * p.C + p.g_q0[g] + r;
    uint4 o;
    o.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    o.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    o.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    o.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4*>(p.out + (tok * p.nq + h) * p.hd + part8 * 8) = o;
    if (part8 == 0 && p.lse != nullptr) p.lse[tok * p.nq + h] = m + __logf(wsum);
  }
}

}  // namespace cpattn
