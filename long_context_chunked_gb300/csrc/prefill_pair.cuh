// The fused chunked-prefill kernel on PAIRS of SMs with 2-SM MMAs
// (tcgen05 cta_group::2): the same single-pass algorithm as prefill.cuh (one
// query chunk against its cached prefix and its own causal chunk, one online
// softmax -- PCP ring-cache PR, Summary and Design sections), with the two
// CTAs of a cluster working on two adjacent q heads of ONE kv head, i.e. on
// the same K/V tiles.
//
// The leader CTA (cluster rank 0) issues every MMA for both:
//   S[256 x 128]  = Q[256 x HD] K^T   rows 0-127: the leader's head, 128-255:
//                                     the peer's; each CTA holds its own Q and
//                                     64 of the tile's 128 keys (B split by N)
//   O[256 x HD]  += P[256 x 128] V    P from each CTA's own TMEM; each CTA
//                                     holds HD/2 of V's columns (B split by N)
// so each SM stages HALF of every K and V tile (64 KB at HD = 256 instead of
// 128 KB) and the same 16 KB-slot ring holds twice as many tiles.  TMEM use,
// the softmax and the epilogue are those of the single-CTA kernel, per CTA.
//
// Ring slot contents (16 KB, 128-byte swizzle, boxes of 64 columns x 64 rows):
//   K slot j:  chunks 2j, 2j+1 of this CTA's 64 key rows   (HD/128 slots)
//   V slot j:  key rows [j*VR, j*VR + VR) x this CTA's HD/2 columns, one box
//              per 64-column chunk (VR = 16384/HD rows)      (HD/128 slots)
//
// Barriers (per CTA; the leader's are the ones waited on):
//   Q_FULL, SLOT_FULL  on the leader, count 2: one expect_tx arrival from each
//                      CTA's producer; the bytes of both CTAs' copies complete
//                      on them (cta_group::2 TMA)
//   P_FULL             on the leader, count 16: one arrival per softmax warp
//                      of both CTAs
//   S_FULL, O_DONE, SLOT_EMPTY, Q_EMPTY   in both CTAs, count 1: multicast
//                      commits of the leader's MMA thread
#pragma once

#include "prefill.cuh"

namespace cpattn {

template <int HD>
struct PairLayout {
  static constexpr int KSLOTS = HD / 128;      // K half-tile slots per tile
  static constexpr int VSLOTS = HD / 128;      // V half-tile slots per tile
  static constexpr int NH = HD / 2;            // V columns held by one CTA
  static constexpr int VR = 16384 / HD;        // key rows per V slot
  static constexpr int VCH = NH / 64;          // 64-column boxes per V slot row group
  static constexpr int VRG = VR / 64;          // 64-row boxes per V slot column chunk
  static constexpr int BOX = 8192;             // bytes per 64 x 64 box
  static constexpr uint32_t IDESC_QK = make_idesc_bf16(2 * kBQ, kBKV, false);
  static constexpr uint32_t IDESC_PV = make_idesc_bf16(2 * kBQ, HD, true);
  static constexpr uint32_t IDESC_PV_F16 = make_idesc_f16(2 * kBQ, HD, true);
  // One arrival per softmax warp of both CTAs that takes the tile.
  static constexpr uint32_t P_ARRIVALS = 2 * Layout<HD>::P_THREADS / 32;
  static_assert(VCH * VRG * BOX == Layout<HD>::SUB, "V slot = 16 KB");
  static_assert(2 * BOX == Layout<HD>::SUB, "K slot = two chunks of 64 rows");
};

// ------------------------------------------------------------- TMA producer
// Both CTAs: this CTA's half of every K and V tile, and its own Q, each copy
// completing on the leader's barrier.
template <int HD>
__device__ __forceinline__ void producer_role_pair2(const PrefillParams& p, uint32_t sbase,
                                                    const BoundedWait& wait) {
  using Ly = Layout<HD>;
  using Pl = PairLayout<HD>;
  auto bar = [&](int i) { return sbase + Ly::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  const uint32_t rank = cluster_ctarank();
  auto lead = [&](int i) { return mapa_shared(bar(i), 0); };
  RingPos rp;
  long long issued = 0;
  uint32_t q_issued = 0;
  bool ok = true;

  // One slot: wait until both CTAs' last use of it completed (the leader's
  // MMAs released it), announce 16 KB on the leader's full barrier, then
  // issue this CTA's boxes (emit(dst) issues them).
  auto load_slot = [&](auto&& emit) {
    if (rp.round && !wait(bar(Ly::B_SLOTEMPTY + rp.slot), rp.phase ^ 1u, kSiteSlotEmpty))
      return false;
    const uint32_t full = lead(Ly::B_SLOTFULL + rp.slot);
    count_arrive(p.bar_counts, 1u, Ly::B_SLOTFULL + rp.slot, 1);
    mbar_arrive_expect_tx_remote(full, Ly::SUB);
    emit(sbase + Ly::OFF_RING + static_cast<uint32_t>(rp.slot) * Ly::SUB, full);
    rp.template advance<Ly::NSLOT>();
    ++issued;
    return true;
  };

  for (int ur = 0, u = unit_of<2>(0); ok && u < p.num_units; u = unit_of<2>(++ur)) {
    const Unit U = decode_unit(p, u);
    if (q_issued > 0 && !wait(bar(Ly::B_QEMPTY), (q_issued - 1) & 1u, kSiteQEmpty)) {
      ok = false;
      break;
    }
    const uint32_t qfull = lead(Ly::B_QFULL);
    count_arrive(p.bar_counts, 1u, Ly::B_QFULL, 1);
    mbar_arrive_expect_tx_remote(qfull, Ly::Q_BYTES);
    for (int c = 0; c < Ly::KCH; ++c)
      tma_load_3d_pair(sbase + Ly::OFF_Q + c * (kBQ * 128), &p.tm_q, qfull, 64 * c, U.h,
                       U.b * p.C + U.q0);
    ++q_issued;

    const int head_row = ((U.b * p.nkv + U.g) * p.P) * p.S;
    CacheWalk wk, wv;
    wk.init(U.L, p.P, p.S);
    wv.init(U.L, p.P, p.S);
    // Tile v's source is chosen by value, as in the single-CTA producer.
    auto load_k = [&](int v) {
      const bool in_cache = v < U.n_cache;
      const int tile = in_cache ? wk.next() : 0;
      const CUtensorMap* m = in_cache ? &p.tm_k_cache_h : &p.tm_k_new_h;
      const int y = in_cache ? 0 : U.g;
      const int z = (in_cache ? head_row + tile * kBKV : U.b * p.C + (v - U.n_cache) * kBKV) +
                    static_cast<int>(rank) * (kBKV / 2);
      for (int j = 0; j < Pl::KSLOTS; ++j) {
        const bool r = load_slot([&](uint32_t dst, uint32_t full) {
          tma_load_3d_pair(dst, m, full, 64 * (2 * j), y, z);
          tma_load_3d_pair(dst + Pl::BOX, m, full, 64 * (2 * j + 1), y, z);
        });
        if (!r) return false;
      }
      return true;
    };
    auto load_v = [&](int v) {
      const bool in_cache = v < U.n_cache;
      const int tile = in_cache ? wv.next() : 0;
      const CUtensorMap* m = in_cache ? &p.tm_v_cache_h : &p.tm_v_new_h;
      const int y = in_cache ? 0 : U.g;
      const int z = in_cache ? head_row + tile * kBKV : U.b * p.C + (v - U.n_cache) * kBKV;
      const int x0 = static_cast<int>(rank) * Pl::NH;
      for (int j = 0; j < Pl::VSLOTS; ++j) {
        const bool r = load_slot([&](uint32_t dst, uint32_t full) {
          for (int i = 0; i < Pl::VCH; ++i)
            for (int g = 0; g < Pl::VRG; ++g)
              tma_load_3d_pair(dst + (i * Pl::VRG + g) * Pl::BOX, m, full, x0 + 64 * i, y,
                               z + j * Pl::VR + 64 * g);
        });
        if (!r) return false;
      }
      return true;
    };
    // This block's slice of the walk starts at virtual tile U.v0.
    const int skip = U.v0 < U.n_cache ? U.v0 : U.n_cache;
    wk.skip(skip);
    wv.skip(skip);
    // Same order as the MMA consumes them: K0, (K1, V0), (K2, V1), ..., V_last.
    const int v0 = U.v0, v1 = U.v0 + U.n_tiles;
    ok = load_k(v0);
    for (int v = v0 + 1; ok && v < v1; ++v) ok = load_k(v) && load_v(v - 1);
    if (ok) ok = load_v(v1 - 1);
  }

  if (!ok && rank == 0) {
    // The leader's full barriers count both CTAs' copies: let every phase
    // the leader took part in land before the pair can leave (bounded; a
    // phase the peer never joined gives up after the drain limit).
    const long long first = issued > Ly::NSLOT ? issued - Ly::NSLOT : 0;
    for (long long z = first; z < issued; ++z)
      mbar_wait_drain(bar(Ly::B_SLOTFULL + static_cast<int>(z % Ly::NSLOT)),
                      static_cast<uint32_t>((z / Ly::NSLOT) & 1), kDrainLimitNs);
    if (q_issued > 0) mbar_wait_drain(bar(Ly::B_QFULL), (q_issued - 1) & 1u, kDrainLimitNs);
  }
}

// ------------------------------------------------------------- MMA issuer
// Leader CTA only, the whole MMA warp: control flow and operands are
// warp-uniform (every wait's outcome is agreed by the warp), and each MMA and
// commit is issued by one elected lane.
template <int HD, bool SPLIT, int VF16>
__device__ __forceinline__ void mma_role_pair2(const PrefillParams& p, uint32_t sbase,
                                               uint32_t tmem, const BoundedWait& wait) {
  using Ly = Layout<HD>;
  using Pl = PairLayout<HD>;
  auto bar = [&](int i) { return sbase + Ly::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  const uint32_t q_base = sbase + Ly::OFF_Q;
  const uint32_t ring = sbase + Ly::OFF_RING;
  // Operand descriptors are a base's descriptor plus (offset >> 4): the
  // start-address field holds address >> 4 in 14 bits, and every offset
  // stays inside its buffer (Q, or one ring slot), so the sum never carries.
  // Fewer instructions in the MMA warp, which shares a sub-partition with
  // two softmax warps.
  const uint64_t qdesc = make_sdesc_sw128(q_base, 16, 1024);
  RingPos rp;
  uint32_t tile_ctr = 0, units = 0;
  bool ok = true;
  auto wwait = [&](uint32_t b, uint32_t parity, int site) {
    return __all_sync(0xFFFFFFFFu, wait(b, parity, site));
  };
  // Commit of the leader's MMAs so far, arriving on barrier i of the CTAs in
  // cta_mask (0x3: both, 0x1: the leader).
  auto commit = [&](int i, uint16_t cta_mask) {
    count_commit(p.bar_counts, cta_mask, i);
    mma2_commit_mc(bar(i), cta_mask);
  };
#ifdef CPATTN_SERIALIZE_MMA
  // Race-detection build: every MMA group completes before the MMA thread
  // moves on (see prefill.cuh).
  uint32_t ser_phase = 0;
  auto serialize = [&]() {
    commit(Ly::B_DRAIN, 0x1);
    mbar_wait_drain(bar(Ly::B_DRAIN), ser_phase, kDrainLimitNs);
    count_wait(p.bar_counts, kCountRowMma, Ly::B_DRAIN);
    ser_phase ^= 1u;
  };
#else
  auto serialize = []() {};
  const uint32_t ser_phase = 0;
#endif

  // O (+)= P_w V_w over both CTAs' rows, P_w from the S buffer of tile t;
  // F16: a tile of the fp16 V cache (one product of fp16 P and V per 16
  // keys).  The form is chosen once per tile: a branch between the elected
  // MMAs of the warp would cost every MMA a reconvergence.
  auto issue_pv_as = [&](int w, uint32_t t, auto f16tag) {
    constexpr bool F16 = decltype(f16tag)::value;
    const uint32_t sb = t & 1u;
    if (!wwait(bar(Ly::B_PFULL + sb), (t >> 1) & 1u, kSitePFull)) return false;
    tc_fence_after();
    const uint32_t p_tmem = tmem + HD + sb * kBKV;
    // SPLIT_O: tile t accumulates into O_{t % 2} (see prefill.cuh).
    const uint32_t o_tmem = tmem + (Ly::SPLIT_O && sb ? Ly::O_COL1 : 0u);
    const int w_acc = Ly::SPLIT_O ? (w >> 1) : w;
    for (int j = 0; j < Pl::VSLOTS; ++j) {
      if (!wwait(bar(Ly::B_SLOTFULL + rp.slot), rp.phase, kSiteSlotFull)) return false;
      tc_fence_after();
      const uint32_t vb = ring + static_cast<uint32_t>(rp.slot) * Ly::SUB;
      const uint64_t vdesc = make_sdesc_sw128(vb, Pl::VR * 128, 1024);
#pragma unroll
      for (int kk = 0; kk < Pl::VR / 16; ++kk) {
        // V: VCH column chunks of VR rows x 128 B (chunk stride VR * 128),
        // 16 key rows per step.
        const uint64_t bd = vdesc + static_cast<uint64_t>((kk * 2048) >> 4);
        const int e0 = j * Pl::VR + kk * 16;
        const uint32_t pa = p_tmem + 32 * (e0 >> 5) + ((e0 & 31) >> 1);
        if (F16) {
          mma2_ts(o_tmem, pa, bd, Pl::IDESC_PV_F16, (w_acc | j | kk) != 0);
        } else {
          mma2_ts(o_tmem, pa, bd, Pl::IDESC_PV, (w_acc | j | kk) != 0);
          if (SPLIT) mma2_ts(o_tmem, pa + 16, bd, Pl::IDESC_PV, 1u);
        }
      }
      serialize();
      commit(Ly::B_SLOTEMPTY + rp.slot, 0x3);
      rp.template advance<Ly::NSLOT>();
    }
    commit(Ly::B_ODONE + static_cast<int>(t & 1u), 0x3);
    return true;
  };
  auto issue_pv = [&](const Unit& U, int w, uint32_t t) {
    if constexpr (VF16) {
      if (VF16 == kVF16All || U.v0 + w < U.n_cache) return issue_pv_as(w, t, std::true_type{});
    }
    return issue_pv_as(w, t, std::false_type{});
  };

  for (int ur = 0, u = unit_of<2>(0); ok && u < p.num_units; u = unit_of<2>(++ur), ++units) {
    const Unit U = decode_unit(p, u);
    if (!wwait(bar(Ly::B_QFULL), units & 1u, kSiteQFull)) {
      ok = false;
      break;
    }
    tc_fence_after();
    for (int v = 0; v < U.n_tiles; ++v) {
      const uint32_t sb = tile_ctr & 1u;
      const uint32_t s_tmem = tmem + HD + sb * kBKV;
      for (int j = 0; j < Pl::KSLOTS; ++j) {
        if (!wwait(bar(Ly::B_SLOTFULL + rp.slot), rp.phase, kSiteSlotFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kb = ring + static_cast<uint32_t>(rp.slot) * Ly::SUB;
        const uint64_t kdesc = make_sdesc_sw128(kb, 16, 1024);
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int c = 2 * j + c2;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = qdesc + static_cast<uint64_t>((c * (kBQ * 128) + kk * 32) >> 4);
            const uint64_t bd = kdesc + static_cast<uint64_t>((c2 * Pl::BOX + kk * 32) >> 4);
            mma2_ss(s_tmem, ad, bd, Pl::IDESC_QK, (c | kk) != 0);
          }
        }
        serialize();
        commit(Ly::B_SLOTEMPTY + rp.slot, 0x3);
        rp.template advance<Ly::NSLOT>();
      }
      if (!ok) break;
      commit(Ly::B_SFULL + sb, 0x3);
      if (v == U.n_tiles - 1) commit(Ly::B_QEMPTY, 0x3);
      if (v >= 1 && !issue_pv(U, v - 1, tile_ctr - 1)) {
        ok = false;
        break;
      }
      ++tile_ctr;
    }
    if (ok) ok = issue_pv(U, U.n_tiles - 1, tile_ctr - 1);
  }
  // Every MMA issued must complete before either CTA releases its TMEM.
  commit(Ly::B_DRAIN, 0x1);
  if (mbar_wait_drain(bar(Ly::B_DRAIN), ser_phase, kDrainLimitNs))
    count_wait(p.bar_counts, kCountRowMma, Ly::B_DRAIN);
}

// ------------------------------------------------------------------ kernel
// Launched with clusters of two CTAs; CTA 2k + r runs units 2s + r of each
// round of gridDim.x units (s = k in even rounds, E - 1 - k in odd ones:
// unit_of), so the pair always holds q heads 2i and 2i + 1 of the same row
// block (the host launches it only when the group size is even).
template <int HD, bool SPLIT, int VF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel_pair2(const __grid_constant__ PrefillParams p) {
  using Ly = Layout<HD>;
  using Pl = PairLayout<HD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  // Same base offset in both CTAs (same kernel), so both leave here together.
  if (sbase - raw > static_cast<uint32_t>(Ly::ALIGN_SLACK)) {
    if (threadIdx.x == 0 && p.status != nullptr) atomicCAS(p.status, kStatusOk, kStatusLayout);
    return;
  }
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Ly::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  auto bar = [&](int i) { return sbase + Ly::OFF_BAR + 8u * static_cast<uint32_t>(i); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < Ly::NBAR; ++i) {
      uint32_t count = 1;
      if (i == Ly::B_QFULL || (i >= Ly::B_SLOTFULL && i < Ly::B_SLOTEMPTY)) count = 2;
      if (i == Ly::B_PFULL || i == Ly::B_PFULL + 1) count = Pl::P_ARRIVALS;
      mbar_init(bar(i), count);
    }
    *abort_flag = 0;
    for (int i = 0; i < 4; ++i) reinterpret_cast<volatile int*>(smem + Ly::OFF_PFAIL)[i] = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_k_new_h);
    prefetch_tmap(&p.tm_k_cache_h);
    prefetch_tmap(&p.tm_v_new_h);
    prefetch_tmap(&p.tm_v_cache_h);
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(smem_u32(tmem_holder), Ly::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  // Both CTAs' barriers are initialised before any copy or arrival crosses.
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const BoundedWait wait = make_wait(abort_flag, p, bar(0), warp);

  if (warp < kProducerWarp) {
    if constexpr (Ly::SPLIT_O) {
      reg_alloc_inc<kSoftmaxRegs>();
      softmax_role_rows<SPLIT, true, VF16, 2>(p, sbase, tmem, wait);
    } else {
      softmax_role<HD, SPLIT, true, VF16, 2>(p, sbase, tmem, wait);
    }
  } else {
    if constexpr (Ly::SPLIT_O) reg_alloc_dec<kOtherRegs>();
    if (warp == kProducerWarp) {
      if (lane == 0) {
        // The staged fp16 V is written by the kernel this one depends on.
        if constexpr (VF16 == kVF16All) griddep_wait();
        producer_role_pair2<HD>(p, sbase, wait);
      }
    } else if (warp == kWriterWarp) {
      if (p.k_cache_w != nullptr) kv_write_lanes<HD, VF16 != kVBf16, 2>(p, lane);
    } else if (warp == kMmaWarp && rank == 0) {
      mma_role_pair2<HD, SPLIT, VF16>(p, sbase, tmem, wait);
    }
  }
  __syncwarp();
  tc_fence_before();
  // The leader's MMAs (which write both CTAs' TMEM) have drained and both
  // CTAs' softmax warps are done with TMEM before either CTA releases it.
  cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, Ly::TMEM_COLS);
  }
  // Neither CTA leaves while the other may still arrive on its barriers.
  cluster_sync();
}

}  // namespace cpattn
