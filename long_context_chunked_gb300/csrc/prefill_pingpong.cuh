// The fused chunked-prefill kernel with TWO query tiles per CTA (HD = 128):
// the same single-pass algorithm as prefill.cuh (one query chunk against its
// cached prefix and its own causal chunk, one online softmax -- PCP
// ring-cache PR, Summary and Design sections), with one CTA working on two
// adjacent q heads of ONE kv head, i.e. on the same K/V tiles, and one
// warpgroup of softmax warps per head.
//
// Why: at HD = 128 a tile's two products (QK^T and P.V) are short next to
// the softmax of the tile, and with one query tile the tensor core waits for
// every softmax.  With two, the tensor core runs one tile's products while
// the other tile's softmax runs:
//
//   MMA:      PV_A(v-1)  QK_A(v)  PV_B(v-1)  QK_B(v)  PV_A(v)  QK_A(v+1) ...
//   softmax A:                    [---- S_A(v) -> P_A(v) ----]
//   softmax B:  [-- S_B(v-1) -> P_B(v-1) --]          [---- S_B(v) -> ...
//
// Each K and V tile in shared memory serves both heads, so every SM stages
// half the K/V bytes per product that a one-head CTA does (as the 2-SM pair
// kernel does across two SMs).
//
// TMEM (512 columns): O_A [0, 128), O_B [128, 256), S/P_A [256, 384), S/P_B
// [384, 512).  A query tile has ONE S buffer: QK_A(v+1) overwrites P_A(v),
// so it is issued after PV_A(v); the tensor pipe runs one CTA's MMAs in
// issue order.  The same order lets the softmax rescale O_A while it holds
// tile v: the S_FULL_A commit of tile v follows PV_A(v-1), so every earlier
// product into O_A has completed when S_A(v) is ready.
//
// Each softmax warp holds 32 whole rows of its tile (all 128 columns), so
// the row max needs no exchange between warps.
//
// Ring order (16 KB slots): K(0), V(0), K(1), V(1), ...; the MMA warp uses
// V(v-1) then K(v) at step v, each twice (A, then B), and releases a slot
// after its second use.
//
// Barriers (count 1 unless noted): Q_FULL, Q_EMPTY; S_FULL[tile],
// P_FULL[tile] (count 4: one arrival per softmax warp of the tile),
// O_DONE[tile] (once per unit pair); SLOT_FULL/EMPTY[NSLOT]; DRAIN.
#pragma once

#include "prefill.cuh"

namespace cpattn {

struct PingPongLayout {
  static constexpr int HD = 128;
  static constexpr int KCH = HD / 64;            // 64-column chunks per row (one K slot each)
  static constexpr int VROWS = 8192 / HD;        // kv rows per V slot (16 KB)
  static constexpr int VSUB = kBKV / VROWS;      // V slots per tile
  static constexpr int SUB = 16384;              // bytes per ring slot
  static constexpr int Q_BYTES = kBQ * HD * 2;   // one query tile
  static constexpr int NSLOT = 10;
  static constexpr int OFF_Q = 0;                // tile A, then tile B
  static constexpr int OFF_RING = 2 * Q_BYTES;
  static constexpr int OFF_BAR = OFF_RING + NSLOT * SUB;
  // S_FULL, P_FULL and O_DONE: one barrier per query tile (+0: A, +1: B).
  static constexpr int B_QFULL = 0, B_QEMPTY = 1, B_SFULL = 2, B_PFULL = 4, B_ODONE = 6,
                       B_DRAIN = 8, B_SLOTFULL = 9, B_SLOTEMPTY = 9 + NSLOT;
  static constexpr int NBAR = 9 + 2 * NSLOT;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int ALIGN_SLACK = 512;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + ALIGN_SLACK;
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t O_COL = 0;           // + tile * HD
  static constexpr uint32_t S_COL = 2 * HD;      // + tile * kBKV
  static constexpr uint32_t P_ARRIVALS = kSoftmaxWarps / 2;
  static constexpr uint32_t IDESC_QK = make_idesc_bf16(kBQ, kBKV, false);
  static constexpr uint32_t IDESC_PV = make_idesc_bf16(kBQ, HD, true);
  static constexpr uint32_t IDESC_PV_F16 = make_idesc_f16(kBQ, HD, true);
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(2 * HD + 2 * kBKV <= TMEM_COLS, "TMEM budget");
  static_assert(kSoftmaxWarps == 8, "one warpgroup of softmax warps per query tile");
};

// Unit k (0: tile A, 1: tile B) of this CTA's r-th round.  A CTA takes the
// unit pairs (2j, 2j + 1) -- two q heads of one kv head and one row block --
// dealt in the boustrophedon order of unit_of.
__device__ __forceinline__ int unit_pingpong(int r, int k) {
  const int E = static_cast<int>(gridDim.x);
  const int e = static_cast<int>(blockIdx.x);
  const int slot = (r & 1) ? E - 1 - e : e;
  return (r * E + slot) * 2 + k;
}

// ------------------------------------------------------------- TMA producer
__device__ __forceinline__ void producer_role_pingpong(const PrefillParams& p, uint32_t sbase,
                                                       const BoundedWait& wait) {
  using Ly = PingPongLayout;
  auto bar = [&](int i) { return sbase + Ly::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  RingPos rp;
  long long issued = 0;
  uint32_t q_issued = 0;
  bool ok = true;

  // One slot: wait until it is free, expect 16 KB, issue `nbox` boxes of
  // `box` bytes (64 columns each, from column x0).
  auto load_slot = [&](const CUtensorMap* m, int nbox, int box, int x0, int y, int z) {
    if (rp.round && !wait(bar(Ly::B_SLOTEMPTY + rp.slot), rp.phase ^ 1u, kSiteSlotEmpty))
      return false;
    const uint32_t full = bar(Ly::B_SLOTFULL + rp.slot);
    count_arrive(p.bar_counts, 1u, Ly::B_SLOTFULL + rp.slot, 1);
    mbar_arrive_expect_tx(full, Ly::SUB);
    const uint32_t dst = sbase + Ly::OFF_RING + static_cast<uint32_t>(rp.slot) * Ly::SUB;
    for (int i = 0; i < nbox; ++i) tma_load_3d(dst + i * box, m, full, x0 + 64 * i, y, z);
    rp.template advance<Ly::NSLOT>();
    ++issued;
    return true;
  };

  for (int ur = 0, u = unit_pingpong(0, 0); ok && u < p.num_units; u = unit_pingpong(++ur, 0)) {
    const Unit U = decode_unit(p, u);  // tile A's unit; tile B's is head U.h + 1
    if (q_issued > 0 && !wait(bar(Ly::B_QEMPTY), (q_issued - 1) & 1u, kSiteQEmpty)) {
      ok = false;
      break;
    }
    count_arrive(p.bar_counts, 1u, Ly::B_QFULL, 1);
    mbar_arrive_expect_tx(bar(Ly::B_QFULL), 2 * Ly::Q_BYTES);
    for (int t = 0; t < 2; ++t)
      for (int c = 0; c < Ly::KCH; ++c)
        tma_load_3d(sbase + Ly::OFF_Q + t * Ly::Q_BYTES + c * (kBQ * 128), &p.tm_q,
                    bar(Ly::B_QFULL), 64 * c, U.h + t, U.b * p.C + U.q0);
    ++q_issued;

    const int head_row = ((U.b * p.nkv + U.g) * p.P) * p.S;
    CacheWalk wk, wv;
    wk.init(U.L, p.P, p.S);
    wv.init(U.L, p.P, p.S);
    const int skip = U.v0 < U.n_cache ? U.v0 : U.n_cache;
    wk.skip(skip);
    wv.skip(skip);
    // Tile v's source is chosen by value: cache map and shard-walk row, or
    // the chunk's token-order map and row.
    for (int v = U.v0; ok && v < U.v0 + U.n_tiles; ++v) {
      const bool in_cache = v < U.n_cache;
      const int y = in_cache ? 0 : U.g;
      const int zk = in_cache ? head_row + wk.next() * kBKV : U.b * p.C + (v - U.n_cache) * kBKV;
      const int zv = in_cache ? head_row + wv.next() * kBKV : U.b * p.C + (v - U.n_cache) * kBKV;
      // K: one 64-column box of 128 rows per slot; V: VROWS rows of all
      // columns per slot, one box per 64 columns.
      for (int c = 0; ok && c < Ly::KCH; ++c)
        ok = load_slot(in_cache ? &p.tm_k_cache : &p.tm_k_new, 1, 0, 64 * c, y, zk);
      for (int j = 0; ok && j < Ly::VSUB; ++j)
        ok = load_slot(in_cache ? &p.tm_v_cache : &p.tm_v_new, Ly::KCH, Ly::VROWS * 128, 0, y,
                       zv + j * Ly::VROWS);
    }
  }

  if (!ok) {
    // Let copies already issued land before this CTA can exit.
    const long long first = issued > Ly::NSLOT ? issued - Ly::NSLOT : 0;
    for (long long z = first; z < issued; ++z)
      mbar_wait_drain(bar(Ly::B_SLOTFULL + static_cast<int>(z % Ly::NSLOT)),
                      static_cast<uint32_t>((z / Ly::NSLOT) & 1), kDrainLimitNs);
    if (q_issued > 0) mbar_wait_drain(bar(Ly::B_QFULL), (q_issued - 1) & 1u, kDrainLimitNs);
  }
}

// ------------------------------------------------------------- MMA issuer
// Run by the whole MMA warp (operands and control flow warp-uniform; each
// MMA and commit is issued by one elected lane).
template <bool SPLIT, int VF16>
__device__ __forceinline__ void mma_role_pingpong(const PrefillParams& p, uint32_t sbase,
                                                  uint32_t tmem, const BoundedWait& wait) {
  using Ly = PingPongLayout;
  constexpr int HD = Ly::HD;
  auto bar = [&](int i) { return sbase + Ly::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  const uint32_t ring = sbase + Ly::OFF_RING;
  RingPos rp;
  uint32_t tile_ctr = 0, units = 0;
  bool ok = true;
  auto wwait = [&](uint32_t b, uint32_t parity, int site) {
    return __all_sync(0xFFFFFFFFu, wait(b, parity, site));
  };
  auto commit = [&](int i) {
    count_commit(p.bar_counts, 1u, i);
    mma_commit(bar(i));
  };
#ifdef CPATTN_SERIALIZE_MMA
  // Race-detection build: every MMA group completes before the MMA warp
  // moves on (see mma_role).
  uint32_t ser_phase = 0;
  auto serialize = [&]() {
    commit(Ly::B_DRAIN);
    mbar_wait_drain(bar(Ly::B_DRAIN), ser_phase, kDrainLimitNs);
    count_wait(p.bar_counts, kCountRowMma, Ly::B_DRAIN);
    ser_phase ^= 1u;
  };
#else
  auto serialize = []() {};
  const uint32_t ser_phase = 0;
#endif

  // S_q = Q_q K^T over the K tile whose first slot is at rk.  `first`: the
  // tile's first use (waits for its slots), else its second (releases them).
  auto issue_qk = [&](int q, RingPos rk, bool first) {
    const uint32_t s_tmem = tmem + Ly::S_COL + static_cast<uint32_t>(q) * kBKV;
    const uint32_t q_base = sbase + Ly::OFF_Q + static_cast<uint32_t>(q) * Ly::Q_BYTES;
    for (int c = 0; c < Ly::KCH; ++c) {
      if (first) {
        if (!wwait(bar(Ly::B_SLOTFULL + rk.slot), rk.phase, kSiteSlotFull)) return false;
        tc_fence_after();
      }
      const uint32_t kb = ring + static_cast<uint32_t>(rk.slot) * Ly::SUB;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = make_sdesc_sw128(q_base + c * (kBQ * 128) + kk * 32, 16, 1024);
        const uint64_t bd = make_sdesc_sw128(kb + kk * 32, 16, 1024);
        mma_ss(s_tmem, ad, bd, Ly::IDESC_QK, (c | kk) != 0);
      }
      serialize();
      if (!first) commit(Ly::B_SLOTEMPTY + rk.slot);
      rk.template advance<Ly::NSLOT>();
    }
    commit(Ly::B_SFULL + q);
    return true;
  };
  // O_q (+)= P_q V over the V tile whose first slot is at rv, P_q of global
  // tile t; w: the tile's index in the unit (0 overwrites O).  F16: a tile
  // of the fp16 V cache (one product of fp16 P and V per 16 keys).
  auto issue_pv_as = [&](int q, RingPos rv, bool first, int w, uint32_t t, auto f16tag) {
    constexpr bool F16 = decltype(f16tag)::value;
    if (!wwait(bar(Ly::B_PFULL + q), t & 1u, kSitePFull)) return false;
    tc_fence_after();
    const uint32_t p_tmem = tmem + Ly::S_COL + static_cast<uint32_t>(q) * kBKV;
    const uint32_t o_tmem = tmem + Ly::O_COL + static_cast<uint32_t>(q) * HD;
    for (int j = 0; j < Ly::VSUB; ++j) {
      if (first) {
        if (!wwait(bar(Ly::B_SLOTFULL + rv.slot), rv.phase, kSiteSlotFull)) return false;
        tc_fence_after();
      }
      const uint32_t vb = ring + static_cast<uint32_t>(rv.slot) * Ly::SUB;
#pragma unroll
      for (int kk = 0; kk < Ly::VROWS / 16; ++kk) {
        const uint64_t bd = make_sdesc_sw128(vb + kk * 2048, Ly::VROWS * 128, 1024);
        // P of key rows e0..e0+15: chunk e0/32, 8 packed columns at
        // (e0 % 32) / 2 within the chunk's hi half; its lo half follows.
        const int e0 = j * Ly::VROWS + kk * 16;
        const uint32_t pa = p_tmem + 32 * (e0 >> 5) + ((e0 & 31) >> 1);
        if (F16) {
          mma_ts(o_tmem, pa, bd, Ly::IDESC_PV_F16, (w | j | kk) != 0);
        } else {
          mma_ts(o_tmem, pa, bd, Ly::IDESC_PV, (w | j | kk) != 0);
          if (SPLIT) mma_ts(o_tmem, pa + 16, bd, Ly::IDESC_PV, 1u);
        }
      }
      serialize();
      if (!first) commit(Ly::B_SLOTEMPTY + rv.slot);
      rv.template advance<Ly::NSLOT>();
    }
    return true;
  };
  // The P.V form is chosen once per tile: a branch between the elected MMAs
  // of the warp would cost every MMA a reconvergence.
  auto issue_pv = [&](const Unit& U, int q, RingPos rv, bool first, int w, uint32_t t) {
    if constexpr (VF16) {
      if (VF16 == kVF16All || U.v0 + w < U.n_cache)
        return issue_pv_as(q, rv, first, w, t, std::true_type{});
    }
    return issue_pv_as(q, rv, first, w, t, std::false_type{});
  };
  auto skip_slots = [&](int n) {
    for (int i = 0; i < n; ++i) rp.template advance<Ly::NSLOT>();
  };

  for (int ur = 0, u = unit_pingpong(0, 0); ok && u < p.num_units; u = unit_pingpong(++ur, 0), ++units) {
    const Unit U = decode_unit(p, u);
    if (!wwait(bar(Ly::B_QFULL), units & 1u, kSiteQFull)) {
      ok = false;
      break;
    }
    tc_fence_after();
    // Step 0: QK^T of tile 0 for both heads.
    RingPos rk = rp;
    skip_slots(Ly::KCH);
    ok = issue_qk(0, rk, true) && issue_qk(1, rk, false);
    if (ok && U.n_tiles == 1) commit(Ly::B_QEMPTY);
    // Step v: P.V of tile v-1 and QK^T of tile v, alternating the heads.
    for (int v = 1; ok && v < U.n_tiles; ++v) {
      const RingPos rv = rp;
      skip_slots(Ly::VSUB);
      rk = rp;
      skip_slots(Ly::KCH);
      const uint32_t t = tile_ctr + static_cast<uint32_t>(v - 1);
      ok = issue_pv(U, 0, rv, true, v - 1, t) && issue_qk(0, rk, true) &&
           issue_pv(U, 1, rv, false, v - 1, t) && issue_qk(1, rk, false);
      if (ok && v == U.n_tiles - 1) commit(Ly::B_QEMPTY);
    }
    if (!ok) break;
    // Last step: P.V of the last tile; O_DONE[q] completes with it.
    const RingPos rv = rp;
    skip_slots(Ly::VSUB);
    const int w = U.n_tiles - 1;
    const uint32_t t = tile_ctr + static_cast<uint32_t>(w);
    ok = issue_pv(U, 0, rv, true, w, t);
    if (ok) commit(Ly::B_ODONE + 0);
    ok = ok && issue_pv(U, 1, rv, false, w, t);
    if (ok) commit(Ly::B_ODONE + 1);
    tile_ctr += static_cast<uint32_t>(U.n_tiles);
  }
  // Every MMA issued must complete before TMEM is released.
  commit(Ly::B_DRAIN);
  if (mbar_wait_drain(bar(Ly::B_DRAIN), ser_phase, kDrainLimitNs))
    count_wait(p.bar_counts, kCountRowMma, Ly::B_DRAIN);
}

// ------------------------------------------------------- softmax + epilogue
// Warp w holds query tile q = w / 4 and its TMEM lane quarter w % 4: 32 whole
// rows, all kBKV logits of each.
template <bool SPLIT, int VF16>
__device__ __forceinline__ void softmax_role_pingpong(const PrefillParams& p, uint32_t sbase,
                                                      uint32_t tmem, const BoundedWait& wait) {
  using Ly = PingPongLayout;
  constexpr int HD = Ly::HD;
  constexpr int CH = kBKV / 32;  // 32-column TMEM loads per row
  auto bar = [&](int i) { return sbase + Ly::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  const int warp = threadIdx.x >> 5;
  const int q = warp >> 2;                               // query tile
  const int r = ((warp & 3) << 5) | (threadIdx.x & 31);  // row == TMEM lane
  const uint32_t lane_tmem = tmem + (static_cast<uint32_t>(r & ~31) << 16);
  const uint32_t s_tmem = lane_tmem + Ly::S_COL + static_cast<uint32_t>(q) * kBKV;
  const uint32_t o_tmem = lane_tmem + Ly::O_COL + static_cast<uint32_t>(q) * HD;
  const float sl2 = p.scale_log2;
  uint32_t tile_ctr = 0, units = 0;
  bool drop_one = (p.debug_flags & kDebugDropArrive) && blockIdx.x == 0 && threadIdx.x == 0;

  for (int ur = 0, u = unit_pingpong(0, q); u < p.num_units; u = unit_pingpong(++ur, q), ++units) {
    const Unit U = decode_unit(p, u);
    // This row's token (within the chunk); its q head is the unit's.
    const int tok = U.q0 + r;
    CacheWalk walk;
    walk.init(U.L, p.P, p.S);
    walk.skip(U.v0 < U.n_cache ? U.v0 : U.n_cache);
    float m = -INFINITY;  // running reference max of the scaled logits (log2 units)
    float l = 0.f;        // running sum of 2^(x - m)
    bool ok = true;

    for (int v = 0; v < U.n_tiles; ++v) {
      const int va = U.v0 + v;  // virtual tile index within the unit's whole walk
      const bool in_cache = va < U.n_cache;
      uint32_t mw[4];
      if (in_cache) {
        const int tile = walk.next();
        if (walk.last_full) {
          mw[0] = mw[1] = mw[2] = mw[3] = 0xFFFFFFFFu;
        } else {
          walk.column_mask(tile, mw);
        }
      } else {
        // Causal: current tile j holds chunk tokens 128 j .. 128 j + 127; this
        // row sees those <= tok.
        const int lim0 = tok - kBKV * (va - U.n_cache) + 1;
        const int lim = lim0 < 0 ? 0 : (lim0 > kBKV ? kBKV : lim0);
#pragma unroll
        for (int c = 0; c < 4; ++c) mw[c] = causal_word(lim, c);
      }
      const bool need_mask =
          __any_sync(0xFFFFFFFFu, (mw[0] & mw[1] & mw[2] & mw[3]) != 0xFFFFFFFFu);
      ok = __all_sync(0xFFFFFFFFu, wait(bar(Ly::B_SFULL + q), tile_ctr & 1u, kSiteSFull));
      if (!ok) break;
      tc_fence_after();

      // Pass 1: the row's kBKV logits (all TMEM loads in flight together),
      // masked by value, and their max.
      uint32_t rr[CH][32];
#pragma unroll
      for (int c = 0; c < CH; ++c) tmem_ld32_async(s_tmem + 32 * c, rr[c]);
#pragma unroll
      for (int c = 0; c < CH; ++c) tmem_ld32_fence(rr[c]);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < CH; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            rr[c][i] = ((mw[c] >> i) & 1u) ? rr[c][i] : 0xFF800000u;  // -inf
      }
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int c = 0; c < CH; ++c)
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          mx0 = fmaxf(mx0, __uint_as_float(rr[c][i]));
          mx1 = fmaxf(mx1, __uint_as_float(rr[c][i + 1]));
          mx2 = fmaxf(mx2, __uint_as_float(rr[c][i + 2]));
          mx3 = fmaxf(mx3, __uint_as_float(rr[c][i + 3]));
        }
      const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;

      // Lazy rescale: the reference max moves only when a row's new logits
      // exceed it by more than 2^8 (the final O / l is the same either way).
      const float m_new = fmaxf(m, m_tile);
      const bool need = (v > 0) && (m_new > m + 8.f);
      const float alpha = need ? ex2_approx(m - m_new) : 1.f;
      if (v == 0 || need) m = m_new;

      // Pass 2: p = 2^(x - m), its row sum, and P into the tile's S columns.
      const float neg_m = (m == -INFINITY) ? 0.f : -m;
      const float2 sl2x2 = make_float2(sl2, sl2);
      const float2 negm2 = make_float2(neg_m, neg_m);
      float2 lsa = make_float2(0.f, 0.f), lsb = make_float2(0.f, 0.f);
      bool f16_done = false;
      if constexpr (VF16) {
        if (VF16 == kVF16All || in_cache) {
#pragma unroll
          for (int c = 0; c < CH; ++c)
            exp_pack_store<SPLIT, true>(rr[c], s_tmem + 32 * c, sl2x2, negm2, lsa, lsb);
          f16_done = true;
        }
      }
      if (!f16_done) {
#pragma unroll
        for (int c = 0; c < CH; ++c)
          exp_pack_store<SPLIT, false>(rr[c], s_tmem + 32 * c, sl2x2, negm2, lsa, lsb);
      }
      l = l * alpha + ((lsa.x + lsa.y) + (lsb.x + lsb.y));

      // O of this tile's earlier products is complete (see the file head):
      // a row whose reference moved scales it in place.
      if (__any_sync(0xFFFFFFFFu, need)) {
#pragma unroll 1
        for (int ch = 0; ch < HD / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32_wait(o_tmem + 32 * ch, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(o_tmem + 32 * ch, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if ((threadIdx.x & 31) == 0) {
        if (drop_one) {
          drop_one = false;  // fault-injection hook: this arrival never happens
        } else {
          count_arrive(p.bar_counts, 1u, Ly::B_PFULL + q, 1);
          mbar_arrive(bar(Ly::B_PFULL + q));
        }
      }
      ++tile_ctr;
    }
    if (!ok) break;

    // Epilogue: O / l of the unit's rows (valid rows only).
    ok = __all_sync(0xFFFFFFFFu, wait(bar(Ly::B_ODONE + q), units & 1u, kSiteODone));
    if (!ok) break;
    tc_fence_after();
    store_row<HD, HD>(p, U, tok, U.h, 0, o_tmem, m, l, true);
    tc_fence_before();
  }
}

// ------------------------------------------------------------------ kernel
template <bool SPLIT, int VF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel_pingpong(const __grid_constant__ PrefillParams p) {
  using Ly = PingPongLayout;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  if (sbase - raw > static_cast<uint32_t>(Ly::ALIGN_SLACK)) {  // never seen; refuse, do not overrun
    if (threadIdx.x == 0 && p.status != nullptr) atomicCAS(p.status, kStatusOk, kStatusLayout);
    return;
  }
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Ly::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sbase + Ly::OFF_BAR + 8u * static_cast<uint32_t>(i); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < Ly::NBAR; ++i)
      mbar_init(bar(i), (i == Ly::B_PFULL || i == Ly::B_PFULL + 1) ? Ly::P_ARRIVALS : 1u);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_k_new);
    prefetch_tmap(&p.tm_v_new);
    prefetch_tmap(&p.tm_k_cache);
    prefetch_tmap(&p.tm_v_cache);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), Ly::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const BoundedWait wait = make_wait(abort_flag, p, bar(0), warp);

  if (warp < kProducerWarp) {
    softmax_role_pingpong<SPLIT, VF16>(p, sbase, tmem, wait);
  } else if (warp == kProducerWarp) {
    if (lane == 0) {
      // The staged fp16 V is written by the kernel this one depends on.
      if constexpr (VF16 == kVF16All) griddep_wait();
      producer_role_pingpong(p, sbase, wait);
    }
  } else if (warp == kWriterWarp) {
    if (p.k_cache_w != nullptr)
      kv_write_units<Ly::HD, VF16 != kVBf16>(p, lane,
                                             [](int i) { return unit_pingpong(i >> 1, i & 1); });
  } else if (warp == kMmaWarp) {
    mma_role_pingpong<SPLIT, VF16>(p, sbase, tmem, wait);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, Ly::TMEM_COLS);
  }
}

}  // namespace cpattn
