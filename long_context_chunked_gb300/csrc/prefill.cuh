// Fused chunked-prefill attention for sm_103a: cache region and current
// region walked by ONE kernel with ONE online softmax (PCP ring-cache PR,
// Summary and Design sections), on the 5th-generation tensor cores.
//
// Work unit: (sequence b, query head h, q block of 128 rows).  A persistent
// grid of one CTA per SM walks units longest first.  Per unit the CTA runs a
// virtual tile index v over n_cache cache tiles (the striped-shard walk of
// walk.cuh) followed by the causal current tiles 0..qb; the region of tile v
// is selected by the value of one scalar (in_cache = v < n_cache): it picks
// the tensor map and coordinates of the tile loads and the column mask.
//
// Roles (352 threads):
//   warps 0-7  softmax, two warpgroups splitting each row's columns:
//              tcgen05.ld S (32x32b: one row per thread), value mask, online
//              (m, l) update with lazy O rescale, P (bf16) back into TMEM
//              over S's columns, epilogue O / l -> bf16 global stores.
//   warp 8     TMA producer: Q once per unit, then K/V sub-tiles into a ring
//              of 16 KB shared-memory slots.
//   warp 9     TMEM allocation and the MMA issue (the whole warp, one
//              elected lane per instruction):
//              S = Q K^T (both operands in shared memory) and
//              O += P V (P from TMEM, V from shared memory).
//   warp 10    the fused KV write (cpattn_prefill_write_kv), else idle.
//
// TMEM (512 columns x 128 lanes, fp32): O at [0, HD), S double buffer at
// [HD, HD+128) and [HD+128, HD+256).  P_t (bf16, two per column) is written
// over its S buffer, per 32-key chunk over that chunk's own 32 columns: the
// bf16 rounding P_hi of p in the first 16 and, in the accurate mode (SPLIT),
// the bf16 rounding P_lo of the remainder p - P_hi in the next 16; O then
// takes two products P_hi V + P_lo V, which carries p to ~16 bits.  With an
// fp16 V cache (v_f16), cache tiles write P in fp16 instead (11-bit
// significand) and take one product against the fp16 V tile.
// MMAs of one thread execute in issue order, so the QK^T that next
// overwrites that buffer (tile t+2) runs after PV_t read P_t.
#pragma once

#include <type_traits>

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"
#include "walk.cuh"

namespace cpattn {

struct SeqInfo {
  int cache_len, chunk_len, n_cache_tiles, pad;
};

struct PrefillParams {
  CUtensorMap tm_q;        // [T, NQ, HD]       box 64 x 1 x 128
  CUtensorMap tm_k_new;    // [T, NKV, HD]      box 64 x 1 x 128
  CUtensorMap tm_v_new;    // [T, NKV, HD]      box 64 x 1 x VROWS
  CUtensorMap tm_k_cache;  // [rows, 1, HD]     box 64 x 1 x 128
  CUtensorMap tm_v_cache;  // [rows, 1, HD]     box 64 x 1 x VROWS
  CUtensorMap tm_k_new_h;    // as tm_k_new,   box 64 x 1 x 64 (half a tile, paired CTAs)
  CUtensorMap tm_k_cache_h;  // as tm_k_cache, box 64 x 1 x 64
  CUtensorMap tm_v_new_h;    // as tm_v_new,   box 64 x 1 x 64 (2-SM MMA pairs)
  CUtensorMap tm_v_cache_h;  // as tm_v_cache, box 64 x 1 x 64
  CUtensorMap tm_q_packed;   // as tm_q,       box 64 x G x 128/G (GQA-packed units)
  __nv_bfloat16* out;
  float* lse;
  int* status;
  unsigned long long timeout_ns;
  int num_units, nq, nkv, group, P, S, C, debug_flags;
  // Units per work block: unit u is unit (u % per) of block u / per, i.e.
  // q head (or, packed, kv head) hoff + u % per of that block.  Longest-first
  // order: per = NQ (packed: NKV) and hoff = 0.  kv-head-major order (the
  // units that run together read one kv head's K/V, which then stays in L2):
  // one block per (row block, kv head), per = G and hoff = g * G, all of kv
  // head 0's blocks first.
  int per;
  // out_f32: O is written to `out` as fp32 (the two-launch variant's partial
  // results) instead of bf16.
  int out_f32;
  // GQA packing (launches whose chunks are all short): a unit is (sequence,
  // kv head, block of tb = 128 / group tokens) and its 128 rows are (token
  // t0 + r / group, q head g * group + r % group).  0: a unit is (sequence, q
  // head, block of 128 tokens).
  int packed, tb;
  float scale_log2;
  // Fused KV write (null: none): the chunk's K/V rows, read from k_new /
  // v_new, are also copied into the striped caches k_cache_w / v_cache_w.
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  __nv_bfloat16* k_cache_w;
  __nv_bfloat16* v_cache_w;
  // Barrier-count build only: kCountRecord uint32 per CTA (see ptx.cuh), or null.
  uint32_t* bar_counts;
  float* ws_o;    // split-KV pieces: fp32 O / l, [partial rows][NQ][HD]
  float* ws_lse;  // split-KV pieces: LSE, [partial rows][NQ]
  SeqInfo seqs[CPATTN_MAX_SEQS];
  // Work blocks in dealing order.  blocks[i] = (b << 25) | (hoff << 11) |
  // q block (b < 128 sequences, hoff < 16384, q block < 2048);
  // range[i] = (v0 << 16) | v1: the slice [v0, v1) of the block's virtual tile
  // walk (its n_cache cache tiles, then its causal current tiles 0..qb);
  // part[i] = -1 when the block writes the final output, else the first
  // partial row of a split-KV piece (rows q0.. of the block follow it).
  uint32_t blocks[CPATTN_MAX_ROW_BLOCKS];
  uint32_t range[CPATTN_MAX_ROW_BLOCKS];
  int part[CPATTN_MAX_ROW_BLOCKS];
};

enum : int { kDebugDropArrive = 1 };

// Warp roles: 0 .. 4*kColGroups-1 softmax, then the TMA producer, then TMEM +
// MMA.  Softmax warps w and w + 4k (k < kColGroups) hold the same 32 rows
// (TMEM lane quarter w % 4) and split each row's 128 columns between them.
// Two groups (8 softmax warps): four groups measured 3-8 % slower, since the
// softmax is bound by instruction issue, not latency, and every extra warp
// repeats the per-tile scalar work.
constexpr int kColGroups = 2;
constexpr int kSoftmaxWarps = 4 * kColGroups;
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kMmaWarp = kSoftmaxWarps + 1;
// Copies the chunk's K/V into the cache when the KV write is fused into the
// launch; it must not share a warp with the producer or the MMA thread, whose
// waits its copy loop would otherwise serialise (measured: +7-24 % per step).
constexpr int kWriterWarp = kSoftmaxWarps + 2;
// The last warp only completes the third warpgroup (producer, MMA, writer,
// idle), so that registers can move between whole warpgroups (HD = 128).
constexpr int kThreads = 32 * (kSoftmaxWarps + 4);
// Registers per thread: the launch gives every thread kLaunchRegs (the
// __launch_bounds__ cap for kThreads threads, checked on the host before the
// first launch); at HD = 128 the two softmax warpgroups then take
// kSoftmaxRegs and the third warpgroup keeps kOtherRegs -- exactly the
// launch's pool, so the increase never waits for registers nobody frees.
// 208 / 88 rather than 224 / 56: with 56 the MMA and producer roles spill,
// with 200 the softmax does (varlen 3.75 ms at 224 / 56, 3.70 at 208 / 88).
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 208;
constexpr int kOtherRegs = 88;
static_assert(kThreads == 384 && kThreads * kLaunchRegs <= 65536, "one CTA per SM");
static_assert(2 * 128 * kSoftmaxRegs + 128 * kOtherRegs == kThreads * kLaunchRegs,
              "register split = launch allocation");
constexpr uint32_t kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr uint32_t kRowGroupThreads = 32 * kColGroups;  // one named barrier per row group

// V forms of the prefill kernels (template parameter VF16): a bf16 V cache
// (every tile: the bf16 hi + lo P pair, or fast P); an fp16 V cache with the
// chunk's own V read as bf16 V_new (cache tiles: fp16 P and one P.V product;
// current tiles as with a bf16 cache); an fp16 V cache with the chunk's V
// staged in fp16 by the host (tm_v_new, tm_v_new_h point at the staging), so
// that every tile takes fp16 P and one P.V product.
enum : int { kVBf16 = 0, kVF16Cache = 1, kVF16All = 2 };

// Sites recorded in the status word when a bounded wait expires.
enum : int {
  kSiteQEmpty = 1, kSiteSlotEmpty, kSiteQFull, kSiteSlotFull, kSitePFull, kSiteSFull,
  kSiteODone, kSiteDrain
};

template <int HD>
struct Layout {
  static constexpr int KCH = HD / 64;            // 64-column chunks per row (one TMA box each)
  static constexpr int VROWS = 8192 / HD;        // kv rows per V sub-tile (16 KB)
  static constexpr int VSUB = kBKV / VROWS;      // V sub-tiles per tile
  static constexpr int SUB = 16384;              // bytes per ring slot
  static constexpr int Q_BYTES = kBQ * HD * 2;
  static constexpr int NSLOT = HD == 256 ? 10 : 12;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = Q_BYTES;
  static constexpr int OFF_BAR = OFF_RING + NSLOT * SUB;
  // barrier indices
  // O_DONE b completes with every PV of a tile t with t % 2 == b.
  static constexpr int B_QFULL = 0, B_QEMPTY = 1, B_SFULL = 2, B_PFULL = 4, B_ODONE = 6,
                       B_DRAIN = 8, B_SLOTFULL = 9, B_SLOTEMPTY = 9 + NSLOT;
  static constexpr int NBAR = 9 + 2 * NSLOT;
  // HD = 128: two O accumulators, and K/V tiles alternate between the two
  // softmax warpgroups (whole rows per warp; softmax_role_rows).  TMEM:
  // O_0 [0, 128), S_0 [128, 256), S_1 [256, 384), O_1 [384, 512).
  static constexpr bool SPLIT_O = HD == 128;
  static constexpr uint32_t O_COL1 = HD + 2 * kBKV;
  // Softmax arrivals per tile on P_FULL (threads of the warps that take it).
  static constexpr uint32_t P_THREADS = SPLIT_O ? kSoftmaxThreads / 2 : kSoftmaxThreads;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // Row exchange, fp32: [kColGroups][128] maxima (HD = 256); [2][2][128]
  // (m, l) of each warpgroup (HD = 128).
  static constexpr int XCH_FLOATS = SPLIT_O ? 4 * 128 : kColGroups * 128;
  static constexpr int OFF_XCH = OFF_MISC + 16;
  static constexpr int OFF_PFAIL = OFF_XCH + XCH_FLOATS * 4;  // [4] int: a row group gave up
  // Slack for aligning the dynamic shared memory base to 1024 B; the kernel
  // checks at entry that its base needs no more (it is 0 in practice).
  static constexpr int ALIGN_SLACK = 512;
  static constexpr int SMEM_BYTES = OFF_PFAIL + 16 + ALIGN_SLACK;
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t IDESC_QK = make_idesc_bf16(kBQ, kBKV, false);
  static constexpr uint32_t IDESC_PV = make_idesc_bf16(kBQ, HD, true);
  static constexpr uint32_t IDESC_PV_F16 = make_idesc_f16(kBQ, HD, true);
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(HD + 2 * kBKV + (SPLIT_O ? HD : 0) <= TMEM_COLS, "TMEM budget");
};

static_assert(sizeof(PrefillParams) <= 32764, "kernel parameter budget");

struct Unit {
  // h: the q head (packed: the group's first q head); qb: the row block (packed:
  // the token block); q0: its first token.
  int b, h, g, qb, q0, L, c, n_cache;
  int v0, n_tiles;  // this work block's tiles: virtual indices [v0, v0 + n_tiles)
  int part;         // -1, or the first partial row of a split-KV piece
};

__device__ __forceinline__ Unit decode_unit(const PrefillParams& p, int u) {
  Unit U;
  const int per = p.per;
  const int blk = u / per;
  const uint32_t e = p.blocks[blk];
  const int k = static_cast<int>((e >> 11) & 0x3FFFu) + (u - blk * per);
  U.b = static_cast<int>(e >> 25);
  U.qb = static_cast<int>(e & 0x7FFu);
  U.g = p.packed ? k : k / p.group;
  U.h = p.packed ? k * p.group : k;
  U.q0 = U.qb * (p.packed ? p.tb : kBQ);
  U.L = p.seqs[U.b].cache_len;
  U.c = p.seqs[U.b].chunk_len;
  U.n_cache = p.seqs[U.b].n_cache_tiles;
  const uint32_t rg = p.range[blk];
  U.v0 = static_cast<int>(rg >> 16);
  U.n_tiles = static_cast<int>(rg & 0xFFFFu) - U.v0;
  U.part = p.part[blk];
  return U;
}

// The r-th unit of this CTA.  Units are sorted longest first, and they are
// dealt to the executors in boustrophedon order: executor e takes slot e of
// even rounds and slot E-1-e of odd ones.  Dealt cyclically, the same
// executor would take the longest unit of every round; the snake order cuts
// the grid's makespan over the average from 8.4 % to 2.9 % on the 8k
// workload (1.038 -> 1.022 on varlen).  An executor is a CTA, or a cluster
// of `pair` CTAs that take adjacent units (two q heads of one kv head).
// Every role of a CTA walks the same sequence; it ends at the first unit
// index >= num_units (later rounds only hold larger indices).
template <int PAIR>
__device__ __forceinline__ int unit_of(int r) {
  const int E = static_cast<int>(gridDim.x) / PAIR;
  const int e = static_cast<int>(blockIdx.x) / PAIR;
  const int rank = static_cast<int>(blockIdx.x) % PAIR;
  const int slot = (r & 1) ? E - 1 - e : e;
  return r * static_cast<int>(gridDim.x) + slot * PAIR + rank;
}

// The bounded wait of the role that warp `warp` runs (its count row in the
// barrier-count build); bar0 is the shared address of barrier 0.
__device__ __forceinline__ BoundedWait make_wait(volatile int* abort_flag, const PrefillParams& p,
                                                 uint32_t bar0, int warp) {
  const int row = warp < kSoftmaxWarps    ? kCountRowSoftmax
                  : warp == kProducerWarp ? kCountRowProducer
                                          : kCountRowMma;
  return BoundedWait{abort_flag, p.status, p.timeout_ns, p.bar_counts, bar0, row};
}

// Ring position shared by producer and consumer.
struct RingPos {
  int slot = 0;
  uint32_t phase = 0;  // parity of the current use of `slot`
  uint32_t round = 0;  // 0 during the first pass over the ring
  template <int NSLOT>
  __device__ __forceinline__ void advance() {
    if (++slot == NSLOT) {
      slot = 0;
      phase ^= 1u;
      round = 1;
    }
  }
};

}  // namespace cpattn

namespace cpattn {

constexpr unsigned long long kDrainLimitNs = 200ull * 1000 * 1000;

// ------------------------------------------------------------- TMA producer
template <int HD>
__device__ __forceinline__ void producer_role(const PrefillParams& p, uint32_t sbase,
                                              const BoundedWait& wait) {
  using Ly = Layout<HD>;
  auto bar = [&](int i) { return sbase + Ly::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  RingPos rp;
  long long issued = 0;
  uint32_t q_issued = 0;
  bool ok = true;

  // One 16 KB ring slot: wait until the slot is free, expect its 16 KB,
  // then issue its boxes (a K sub-tile is one 64-column box of the 128-row
  // tile; a V sub-tile is KCH boxes of VROWS rows).
  auto load_sub = [&](bool is_k, const CUtensorMap* m, int y, int z, int x0) {
    if (rp.round && !wait(bar(Ly::B_SLOTEMPTY + rp.slot), rp.phase ^ 1u, kSiteSlotEmpty))
      return false;
    const uint32_t full = bar(Ly::B_SLOTFULL + rp.slot);
    count_arrive(p.bar_counts, 1u, Ly::B_SLOTFULL + rp.slot, 1);
    mbar_arrive_expect_tx(full, Ly::SUB);
    const uint32_t dst = sbase + Ly::OFF_RING + static_cast<uint32_t>(rp.slot) * Ly::SUB;
    if (is_k) {
      tma_load_3d(dst, m, full, x0, y, z);
    } else {
      constexpr int BOX = Ly::VROWS * 128;
      for (int i = 0; i < Ly::KCH; ++i) tma_load_3d(dst + i * BOX, m, full, 64 * i, y, z);
    }
    rp.template advance<Ly::NSLOT>();
    ++issued;
    return true;
  };

  for (int ur = 0, u = unit_of<1>(0); ok && u < p.num_units; u = unit_of<1>(++ur)) {
    const Unit U = decode_unit(p, u);
    if (q_issued > 0 && !wait(bar(Ly::B_QEMPTY), (q_issued - 1) & 1u, kSiteQEmpty)) {
      ok = false;
      break;
    }
    count_arrive(p.bar_counts, 1u, Ly::B_QFULL, 1);
    mbar_arrive_expect_tx(bar(Ly::B_QFULL), Ly::Q_BYTES);
    for (int c = 0; c < Ly::KCH; ++c)
      tma_load_3d(sbase + Ly::OFF_Q + c * (kBQ * 128), p.packed ? &p.tm_q_packed : &p.tm_q,
                  bar(Ly::B_QFULL), 64 * c, U.h, U.b * p.C + U.q0);
    ++q_issued;

    const int head_row = ((U.b * p.nkv + U.g) * p.P) * p.S;
    CacheWalk wk, wv;
    wk.init(U.L, p.P, p.S);
    wv.init(U.L, p.P, p.S);
    // Tile v's source is chosen by value: cache map and shard-walk row, or
    // the chunk's token-order map and row.
    auto load_k = [&](int v) {
      const bool in_cache = v < U.n_cache;
      const int tile = in_cache ? wk.next() : 0;
      const CUtensorMap* m = in_cache ? &p.tm_k_cache : &p.tm_k_new;
      const int y = in_cache ? 0 : U.g;
      const int z = in_cache ? head_row + tile * kBKV : U.b * p.C + (v - U.n_cache) * kBKV;
      for (int c = 0; c < Ly::KCH; ++c)
        if (!load_sub(true, m, y, z, 64 * c)) return false;
      return true;
    };
    auto load_v = [&](int v) {
      const bool in_cache = v < U.n_cache;
      const int tile = in_cache ? wv.next() : 0;
      const CUtensorMap* m = in_cache ? &p.tm_v_cache : &p.tm_v_new;
      const int y = in_cache ? 0 : U.g;
      const int z = in_cache ? head_row + tile * kBKV : U.b * p.C + (v - U.n_cache) * kBKV;
      for (int j = 0; j < Ly::VSUB; ++j)
        if (!load_sub(false, m, y, z + j * Ly::VROWS, 0)) return false;
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

  if (!ok) {
    // Let copies already issued land before this CTA can exit.
    const long long first = issued > Ly::NSLOT ? issued - Ly::NSLOT : 0;
    for (long long z = first; z < issued; ++z)
      mbar_wait_drain(bar(Ly::B_SLOTFULL + static_cast<int>(z % Ly::NSLOT)),
                      static_cast<uint32_t>((z / Ly::NSLOT) & 1), kDrainLimitNs);
    if (q_issued > 0) mbar_wait_drain(bar(Ly::B_QFULL), (q_issued - 1) & 1u, kDrainLimitNs);
  }
}

// ------------------------------------------------------- fused KV write
// The writer warp, all 32 lanes.  The unit of
// the first q head of each kv group, in the work block that starts its row
// block's walk (v0 == 0: whole units and first split pieces), copies the row
// block's valid chunk rows of that kv head into the striped caches:
//   cache[b, g, t mod P, t div P, :] = new[b*C + i, g, :],  t = L_b + i
// -- the strided write of write_kv.cuh, so every (token, kv head) is written
// exactly once per launch.  These cache rows hold tokens >= L_b, which no
// unit of this launch reads as keys.  16-byte vectors, consecutive lanes on
// consecutive vectors of a row.  unit_at(i): this CTA's i-th unit.
template <int HD, bool VF16, class UnitAt>
__device__ __forceinline__ void kv_write_units(const PrefillParams& p, int lane, UnitAt unit_at) {
  constexpr int VECS = HD * 2 / 16;  // 16-byte vectors per row
  for (int ur = 0, u = unit_at(0); u < p.num_units; u = unit_at(++ur)) {
    const Unit U = decode_unit(p, u);
    if (U.h % p.group != 0 || U.v0 != 0) continue;
    const int rows = min(p.packed ? p.tb : kBQ, U.c - U.q0);  // valid tokens of the block
    const long long head_row = static_cast<long long>(U.b * p.nkv + U.g) * p.P * p.S;
    for (int i = lane; i < rows * VECS; i += 32) {
      const int r = i / VECS, x = i - r * VECS;
      const int t = U.L + U.q0 + r;
      const long long src = ((static_cast<long long>(U.b) * p.C + U.q0 + r) * p.nkv + U.g) * HD;
      const long long dst = (head_row + static_cast<long long>(t % p.P) * p.S + t / p.P) * HD;
      const uint4 kv = reinterpret_cast<const uint4*>(p.k_new + src)[x];
      uint4 vv = reinterpret_cast<const uint4*>(p.v_new + src)[x];
      if (VF16) {
        bool overflow = false;
        vv = bf16x8_to_f16x8(vv, &overflow);
        if (overflow && p.status != nullptr) atomicCAS(p.status, kStatusOk, kStatusRange);
      }
      reinterpret_cast<uint4*>(p.k_cache_w + dst)[x] = kv;
      reinterpret_cast<uint4*>(p.v_cache_w + dst)[x] = vv;
    }
  }
}

template <int HD, bool VF16, int CL>
__device__ __forceinline__ void kv_write_lanes(const PrefillParams& p, int lane) {
  kv_write_units<HD, VF16>(p, lane, [](int i) { return unit_of<CL>(i); });
}

// ------------------------------------------------------------- MMA issuer
// Run by the whole MMA warp: control flow and operands are warp-uniform (every
// wait's outcome is agreed by the warp), and each MMA and commit is issued by
// one elected lane.
template <int HD, bool SPLIT, int VF16>
__device__ __forceinline__ void mma_role(const PrefillParams& p, uint32_t sbase, uint32_t tmem,
                                         const BoundedWait& wait) {
  using Ly = Layout<HD>;
  auto bar = [&](int i) { return sbase + Ly::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  const uint32_t q_base = sbase + Ly::OFF_Q;
  const uint32_t ring = sbase + Ly::OFF_RING;
  RingPos rp;
  uint32_t tile_ctr = 0, units = 0;
  bool ok = true;
  auto wwait = [&](uint32_t b, uint32_t parity, int site) {
    return __all_sync(0xFFFFFFFFu, wait(b, parity, site));
  };
  // Commit (arrive once on barrier i when every MMA issued so far is done).
  auto commit = [&](int i) {
    count_commit(p.bar_counts, 1u, i);
    mma_commit(bar(i));
  };
#ifdef CPATTN_SERIALIZE_MMA
  // Race-detection build: every MMA group completes before the MMA thread
  // moves on, which stretches the MMA side of every producer/consumer pair.
  // A correct protocol gives the same results bit for bit.
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

  // O (+)= P_w V_w, P_w from the S buffer of global tile t; F16: a tile of
  // the fp16 V cache (one product of fp16 P and V per 16 keys).  The form is
  // chosen once per tile: a branch between the elected MMAs of the warp
  // would cost every MMA a reconvergence.
  auto issue_pv_as = [&](int w, uint32_t t, auto f16tag) {
    constexpr bool F16 = decltype(f16tag)::value;
    const uint32_t sb = t & 1u;
    if (!wwait(bar(Ly::B_PFULL + sb), (t >> 1) & 1u, kSitePFull)) return false;
    tc_fence_after();
    const uint32_t p_tmem = tmem + HD + sb * kBKV;
    // SPLIT_O: tile t accumulates into O_{t % 2}, and the unit's first tile
    // of each parity overwrites it.
    const uint32_t o_tmem = tmem + (Ly::SPLIT_O && sb ? Ly::O_COL1 : 0u);
    const int w_acc = Ly::SPLIT_O ? (w >> 1) : w;
    for (int j = 0; j < Ly::VSUB; ++j) {
      if (!wwait(bar(Ly::B_SLOTFULL + rp.slot), rp.phase, kSiteSlotFull)) return false;
      tc_fence_after();
      const uint32_t vb = ring + static_cast<uint32_t>(rp.slot) * Ly::SUB;
#pragma unroll
      for (int kk = 0; kk < Ly::VROWS / 16; ++kk) {
        // V sub-tile: KCH column chunks of VROWS rows x 128 B, N-contiguous.
        const uint64_t bd = make_sdesc_sw128(vb + kk * 2048, Ly::VROWS * 128, 1024);
        // P of key rows e0..e0+15: chunk e0/32, 8 packed columns at
        // (e0 % 32) / 2 within the chunk's hi half; its lo half follows.
        const int e0 = j * Ly::VROWS + kk * 16;
        const uint32_t pa = p_tmem + 32 * (e0 >> 5) + ((e0 & 31) >> 1);
        if (F16) {
          mma_ts(o_tmem, pa, bd, Ly::IDESC_PV_F16, (w_acc | j | kk) != 0);
        } else {
          mma_ts(o_tmem, pa, bd, Ly::IDESC_PV, (w_acc | j | kk) != 0);
          if (SPLIT) mma_ts(o_tmem, pa + 16, bd, Ly::IDESC_PV, 1u);
        }
      }
      serialize();
      commit(Ly::B_SLOTEMPTY + rp.slot);
      rp.template advance<Ly::NSLOT>();
    }
    commit(Ly::B_ODONE + static_cast<int>(t & 1u));
    return true;
  };
  auto issue_pv = [&](const Unit& U, int w, uint32_t t) {
    if constexpr (VF16) {
      if (VF16 == kVF16All || U.v0 + w < U.n_cache) return issue_pv_as(w, t, std::true_type{});
    }
    return issue_pv_as(w, t, std::false_type{});
  };

  for (int ur = 0, u = unit_of<1>(0); ok && u < p.num_units; u = unit_of<1>(++ur), ++units) {
    const Unit U = decode_unit(p, u);
    if (!wwait(bar(Ly::B_QFULL), units & 1u, kSiteQFull)) {
      ok = false;
      break;
    }
    tc_fence_after();
    for (int v = 0; v < U.n_tiles; ++v) {
      const uint32_t sb = tile_ctr & 1u;
      const uint32_t s_tmem = tmem + HD + sb * kBKV;
      for (int c = 0; c < Ly::KCH; ++c) {
        if (!wwait(bar(Ly::B_SLOTFULL + rp.slot), rp.phase, kSiteSlotFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kb = ring + static_cast<uint32_t>(rp.slot) * Ly::SUB;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = make_sdesc_sw128(q_base + c * (kBQ * 128) + kk * 32, 16, 1024);
          const uint64_t bd = make_sdesc_sw128(kb + kk * 32, 16, 1024);
          mma_ss(s_tmem, ad, bd, Ly::IDESC_QK, (c | kk) != 0);
        }
        serialize();
        commit(Ly::B_SLOTEMPTY + rp.slot);
        rp.template advance<Ly::NSLOT>();
      }
      if (!ok) break;
      commit(Ly::B_SFULL + sb);
      if (v == U.n_tiles - 1) commit(Ly::B_QEMPTY);
      if (v >= 1 && !issue_pv(U, v - 1, tile_ctr - 1)) {
        ok = false;
        break;
      }
      ++tile_ctr;
    }
    if (ok) ok = issue_pv(U, U.n_tiles - 1, tile_ctr - 1);
  }
  // Every MMA issued must complete before TMEM is released.
  commit(Ly::B_DRAIN);
  if (mbar_wait_drain(bar(Ly::B_DRAIN), ser_phase, kDrainLimitNs))
    count_wait(p.bar_counts, kCountRowMma, Ly::B_DRAIN);
}
}  // namespace cpattn

namespace cpattn {

// Column-validity words of a current-region tile for query row r: on the
// diagonal tile key column c is visible iff c <= r (causal, diagonal
// inclusive); tiles left of the diagonal are fully visible.
__device__ __forceinline__ uint32_t causal_word(int lim, int q) {
  const int n = lim - 32 * q;
  return n >= 32 ? 0xFFFFFFFFu : (n <= 0 ? 0u : ((1u << n) - 1u));
}

// p = 2^(x*sl2 - m) over one chunk of 32 logits of a row (x: fp32 bits),
// accumulated into the row sum (lsa: even pairs, lsb: odd pairs) and stored
// as P over the chunk's 32 TMEM columns at taddr: P_hi = bf16(p) in the
// first 16 and, SPLIT, P_lo = bf16(p - P_hi) in the next 16; F16 (a tile of
// an fp16 V cache): fp16(p) in the first 16 (one P.V product).
template <bool SPLIT, bool F16>
__device__ __forceinline__ void exp_pack_store(const uint32_t (&x)[32], uint32_t taddr,
                                               float2 sl2x2, float2 negm2, float2& lsa,
                                               float2& lsb) {
  const float2 minus1 = make_float2(-1.f, -1.f);
  uint32_t hi[16], lo[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 y = __ffma2_rn(
        make_float2(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1])), sl2x2, negm2);
    const float2 pab = make_float2(ex2_approx(y.x), ex2_approx(y.y));
    if (i & 1) lsb = __fadd2_rn(lsb, pab); else lsa = __fadd2_rn(lsa, pab);
    if (F16) {
      hi[i] = pack_f16x2(pab.x, pab.y);
    } else {
      hi[i] = pack_bf16x2(pab.x, pab.y);
      if (SPLIT) {
        const float2 hf = make_float2(__uint_as_float(hi[i] << 16),
                                      __uint_as_float(hi[i] & 0xFFFF0000u));
        const float2 res = __ffma2_rn(hf, minus1, pab);
        lo[i] = pack_bf16x2(res.x, res.y);
      }
    }
  }
  tmem_st16(taddr, hi);
  if (SPLIT && !F16) tmem_st16(taddr + 16, lo);
}

// One output row of a unit from its O columns [ocol0, ocol0 + OCOLS) in
// TMEM (o_tmem: this warp's lanes, column ocol0): a split-KV piece writes
// fp32 O / l and its LSE to its partial rows; a whole unit writes the output
// row (bf16, or fp32 when out_f32).  Rows past the chunk are not written.
// with_lse: this thread also writes the row's LSE, (m + log2 l) ln 2.
template <int HD, int OCOLS>
__device__ __forceinline__ void store_row(const PrefillParams& p, const Unit& U, int row, int head,
                                          int ocol0, uint32_t o_tmem, float m, float l_row,
                                          bool with_lse) {
  const bool valid = row < U.c;
  const float inv_l = 1.f / l_row;
  const bool partial = U.part >= 0;
  const long long tok_g = static_cast<long long>(U.b) * p.C + row;  // token-order row
  const long long orow_i =
      (partial ? static_cast<long long>(U.part + (row - U.q0)) : tok_g) * p.nq + head;
  const bool f32 = partial || p.out_f32 != 0;
  float* lse_out = partial ? p.ws_lse : p.lse;
  uint4* orow = reinterpret_cast<uint4*>(p.out + orow_i * HD + ocol0);
  float4* orow32 = reinterpret_cast<float4*>((partial ? p.ws_o : reinterpret_cast<float*>(p.out)) +
                                             orow_i * HD + ocol0);
#pragma unroll 1
  for (int ch = 0; ch < OCOLS / 32; ++ch) {
    uint32_t o[32];
    tmem_ld32_wait(o_tmem + 32 * ch, o);
    if (valid && f32) {
#pragma unroll
      for (int v4 = 0; v4 < 8; ++v4)
        orow32[ch * 8 + v4] = make_float4(
            __uint_as_float(o[4 * v4]) * inv_l, __uint_as_float(o[4 * v4 + 1]) * inv_l,
            __uint_as_float(o[4 * v4 + 2]) * inv_l, __uint_as_float(o[4 * v4 + 3]) * inv_l);
    } else if (valid) {
#pragma unroll
      for (int v4 = 0; v4 < 4; ++v4) {
        uint4 pk;
        pk.x = pack_bf16x2(__uint_as_float(o[8 * v4 + 0]) * inv_l, __uint_as_float(o[8 * v4 + 1]) * inv_l);
        pk.y = pack_bf16x2(__uint_as_float(o[8 * v4 + 2]) * inv_l, __uint_as_float(o[8 * v4 + 3]) * inv_l);
        pk.z = pack_bf16x2(__uint_as_float(o[8 * v4 + 4]) * inv_l, __uint_as_float(o[8 * v4 + 5]) * inv_l);
        pk.w = pack_bf16x2(__uint_as_float(o[8 * v4 + 6]) * inv_l, __uint_as_float(o[8 * v4 + 7]) * inv_l);
        orow[ch * 4 + v4] = pk;
      }
    }
  }
  if (with_lse && valid && lse_out != nullptr)
    lse_out[orow_i] = (m + __log2f(l_row)) * 0.69314718055994531f;
}

// One output row merged from two partial softmaxes: O = (w0 O_0 + w1 O_1) /
// l_row over the columns [ocol0, ocol0 + OCOLS), O_0 at o0_tmem and O_1 at
// o1_tmem (this warp's lanes); an O whose flag is off is not read (it holds
// no product of this unit).  Outputs as store_row.
template <int HD, int OCOLS>
__device__ __forceinline__ void store_row_merged(const PrefillParams& p, const Unit& U, int row,
                                                 int head, int ocol0, uint32_t o0_tmem,
                                                 uint32_t o1_tmem, float w0, float w1, bool has0,
                                                 bool has1, float m, float l_row, bool with_lse) {
  const bool valid = row < U.c;
  const float inv_l = 1.f / l_row;
  const float a0 = w0 * inv_l, a1 = w1 * inv_l;
  const bool partial = U.part >= 0;
  const long long tok_g = static_cast<long long>(U.b) * p.C + row;
  const long long orow_i =
      (partial ? static_cast<long long>(U.part + (row - U.q0)) : tok_g) * p.nq + head;
  const bool f32 = partial || p.out_f32 != 0;
  float* lse_out = partial ? p.ws_lse : p.lse;
  uint4* orow = reinterpret_cast<uint4*>(p.out + orow_i * HD + ocol0);
  float4* orow32 = reinterpret_cast<float4*>((partial ? p.ws_o : reinterpret_cast<float*>(p.out)) +
                                             orow_i * HD + ocol0);
#pragma unroll 1
  for (int ch = 0; ch < OCOLS / 32; ++ch) {
    // One O buffer at a time through the same 32 registers.
    uint32_t o[32];
    float y[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) y[i] = 0.f;
    if (has0) {
      tmem_ld32_wait(o0_tmem + 32 * ch, o);
#pragma unroll
      for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(o[i]) * a0;
    }
    if (has1) {
      tmem_ld32_wait(o1_tmem + 32 * ch, o);
#pragma unroll
      for (int i = 0; i < 32; ++i) y[i] = fmaf(__uint_as_float(o[i]), a1, y[i]);
    }
    if (valid && f32) {
#pragma unroll
      for (int v4 = 0; v4 < 8; ++v4)
        orow32[ch * 8 + v4] = make_float4(y[4 * v4], y[4 * v4 + 1], y[4 * v4 + 2], y[4 * v4 + 3]);
    } else if (valid) {
#pragma unroll
      for (int v4 = 0; v4 < 4; ++v4) {
        uint4 pk;
        pk.x = pack_bf16x2(y[8 * v4 + 0], y[8 * v4 + 1]);
        pk.y = pack_bf16x2(y[8 * v4 + 2], y[8 * v4 + 3]);
        pk.z = pack_bf16x2(y[8 * v4 + 4], y[8 * v4 + 5]);
        pk.w = pack_bf16x2(y[8 * v4 + 6], y[8 * v4 + 7]);
        orow[ch * 4 + v4] = pk;
      }
    }
  }
  if (with_lse && valid && lse_out != nullptr)
    lse_out[orow_i] = (m + __log2f(l_row)) * 0.69314718055994531f;
}

// ------------------------------------------------------- softmax + epilogue
// kColGroups warpgroups share the 128 rows: warp w reads TMEM lanes
// 32*(w%4).. (its rows) and owns column group h = w/4 of every row -- S
// columns [CW*h, CW*h + CW) with CW = 128 / kColGroups, O columns
// [h*HD/kColGroups, (h+1)*HD/kColGroups).  The kColGroups warps holding the
// same rows (a row group) agree on the row max through one named barrier.
// PAIR2: the CTA is one of a pair whose leader issues 2-SM MMAs; S, P and O
// of this CTA's 128 rows sit in its own TMEM exactly as in a single CTA, but
// "P ready" goes to the leader's barrier, one arrival per warp.
template <int HD, bool SPLIT, bool PAIR2, int VF16, int CL>
__device__ __forceinline__ void softmax_role(const PrefillParams& p, uint32_t sbase, uint32_t tmem,
                                             const BoundedWait& wait) {
  using Ly = Layout<HD>;
  auto bar = [&](int i) { return sbase + Ly::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  constexpr int NG = kColGroups;
  constexpr int CW = kBKV / NG;   // S columns per warp
  constexpr int CH = CW / 32;     // 32-column TMEM loads per warp
  const int warp = threadIdx.x >> 5;
  const int h = warp >> 2;                              // column group
  const int r = ((warp & 3) << 5) | (threadIdx.x & 31);  // row == TMEM lane
  const uint32_t pair_bar = 1u + static_cast<uint32_t>(warp & 3);  // named barrier of the row group
  const uint32_t lane_tmem = tmem + (static_cast<uint32_t>(r & ~31) << 16);
  float* xch = reinterpret_cast<float*>(
      __cvta_shared_to_generic(sbase + Ly::OFF_XCH));   // [NG][128] exchange slots
  // A warp whose bounded wait expired must not leave while the rest of its
  // row group may still reach their barrier: it raises the group's flag and
  // keeps going to the next group barrier, after which all read the flag and
  // leave together.
  volatile int* pair_fail = reinterpret_cast<volatile int*>(
      __cvta_shared_to_generic(sbase + Ly::OFF_PFAIL)) + (warp & 3);
  const float sl2 = p.scale_log2;
  uint32_t tile_ctr = 0;
  bool drop_one = (p.debug_flags & kDebugDropArrive) && blockIdx.x == 0 && threadIdx.x == 0;
  // The wait for the previous tile's P.V before a rescale of O, counted apart
  // from the in-order waits in the barrier-count build.
  const BoundedWait wait_rescale = wait.with_row(kCountRowRescale);
  constexpr int OCOLS = HD / NG;                        // O columns of this group

  for (int ur = 0, u = unit_of<CL>(0); u < p.num_units; u = unit_of<CL>(++ur)) {
    const Unit U = decode_unit(p, u);
    // This row's token (within the chunk) and q head.
    const int tok = U.q0 + (p.packed ? r / p.group : r);
    const int head = p.packed ? U.h + r % p.group : U.h;
    CacheWalk walk;
    walk.init(U.L, p.P, p.S);
    walk.skip(U.v0 < U.n_cache ? U.v0 : U.n_cache);
    float m = -INFINITY;  // running reference max of the scaled logits (log2 units), per row
    float l = 0.f;        // this group's running sum of 2^(x - m)
    bool ok = true;
    bool left_at_vote = false;  // the only way out of the tile loop before its end

    for (int v = 0; v < U.n_tiles; ++v) {
      const int va = U.v0 + v;  // virtual tile index within the unit's whole walk
      const uint32_t sb = tile_ctr & 1u;
      const uint32_t s_tmem = lane_tmem + HD + sb * kBKV + CW * h;

      // Region by value: one scalar picks the validity words of the tile.
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
        for (int q = 0; q < 4; ++q) mw[q] = causal_word(lim, q);
      }
      uint32_t wq[CH];
      uint32_t all_valid = 0xFFFFFFFFu;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int idx = h * CH + c;  // selected by value: no local-memory array
        uint32_t wv = mw[0];
#pragma unroll
        for (int k = 1; k < 4; ++k) wv = (idx == k) ? mw[k] : wv;
        wq[c] = wv;
        all_valid &= wv;
      }
      const bool need_mask = __any_sync(0xFFFFFFFFu, all_valid != 0xFFFFFFFFu);
      // The mask words need no S: they are ready before S is.
      ok = wait(bar(Ly::B_SFULL + sb), (tile_ctr >> 1) & 1u, kSiteSFull);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) *pair_fail = 1;  // decided at the vote below, together with the group
      tc_fence_after();

      // Pass 1: load this group's CW logits (all TMEM loads in flight
      // together), mask by value, and take their max.  The registers stay
      // live for pass 2.
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
            rr[c][i] = ((wq[c] >> i) & 1u) ? rr[c][i] : 0xFF800000u;  // -inf
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
      const float m_half = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;

      // Lazy rescale: the reference max moves only when a row's new logits
      // exceed it by more than 2^8 (the final O / l is the same either way).
      // The row group votes; only then do the groups exchange their maxima.
      float alpha = 1.f;
      bool warp_rescale = false;
      const bool any_need = bar_red_or(pair_bar, kRowGroupThreads,
                                       !ok || *pair_fail != 0 || v == 0 || m_half > m + 8.f);
      if (any_need) {
        if (*pair_fail) {  // read by every warp of the group after the same barrier
          left_at_vote = true;
          break;
        }
        xch[h * 128 + r] = m_half;
        bar_sync(pair_bar, kRowGroupThreads);
        float m_tile = xch[r];
#pragma unroll
        for (int g = 1; g < NG; ++g) m_tile = fmaxf(m_tile, xch[g * 128 + r]);
        const float m_new = fmaxf(m, m_tile);
        const bool need = (v > 0) && (m_new > m + 8.f);
        alpha = need ? ex2_approx(m - m_new) : 1.f;
        warp_rescale = __any_sync(0xFFFFFFFFu, need);
        if (v == 0 || need) m = m_new;
      }

      // Pass 2: p = 2^(x - m) and this group's row sum.  Chunk q (32 keys)
      // holds, over its own 32 columns of the S buffer, P_hi = bf16(p) in the
      // first 16 and -- accurate mode -- P_lo = bf16(p - P_hi) in the next 16.
      const float neg_m = (m == -INFINITY) ? 0.f : -m;
      const float2 sl2x2 = make_float2(sl2, sl2);
      const float2 negm2 = make_float2(neg_m, neg_m);
      float2 lsa = make_float2(0.f, 0.f), lsb = make_float2(0.f, 0.f);
      {
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
      }
      l = l * alpha + ((lsa.x + lsa.y) + (lsb.x + lsb.y));

      // PV completions are observed in order, two tiles behind: PV of tile
      // t-2 on barrier O_DONE[t % 2] (normally complete already: it ran before
      // QK^T of tile t).  A parity wait is unambiguous only while the waiter is
      // at most one phase behind; with the two barriers and PV of tile t held
      // back by this thread's arrival below, that always holds.  Only a tile
      // that rescales O also waits for PV of tile t-1.
      auto pv_wait = [&](const BoundedWait& w, uint32_t t) {
        return w(bar(Ly::B_ODONE + static_cast<int>(t & 1u)), (t >> 1) & 1u, kSiteODone);
      };
      if (tile_ctr >= 2) {
        ok = __all_sync(0xFFFFFFFFu, pv_wait(wait, tile_ctr - 2));
        if (!ok) *pair_fail = 1;  // acted on at the next pair barrier
      }
      if (ok && warp_rescale) {
        ok = __all_sync(0xFFFFFFFFu, pv_wait(wait_rescale, tile_ctr - 1));
        if (!ok) *pair_fail = 1;
        tc_fence_after();
        if (ok) {
#pragma unroll 1
          for (int ch = 0; ch < OCOLS / 32; ++ch) {
            uint32_t o[32];
            tmem_ld32_wait(lane_tmem + h * OCOLS + 32 * ch, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(lane_tmem + h * OCOLS + 32 * ch, o);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      if (PAIR2) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) {
          if (drop_one) {
            drop_one = false;  // fault-injection hook: this arrival never happens
          } else {
            count_arrive(p.bar_counts, 1u, Ly::B_PFULL + sb, 1);  // the leader's barrier
            mbar_arrive_remote(mapa_shared(bar(Ly::B_PFULL + sb), 0));
          }
        }
      } else if (drop_one) {
        drop_one = false;  // fault-injection hook: this arrival never happens
      } else {
        count_arrive(p.bar_counts, 1u, Ly::B_PFULL + sb, 1);
        mbar_arrive(bar(Ly::B_PFULL + sb));
      }
      ++tile_ctr;
    }
    if (left_at_vote) break;  // every warp of the row group left together

    // Epilogue: the row group adds its partial sums (the first barrier keeps
    // the other warps' last reads of the exchange slots ahead of this write,
    // and settles a failure raised after the last vote); each group stores
    // its O columns as bf16 (valid rows only).
    bar_sync(pair_bar, kRowGroupThreads);
    if (*pair_fail) break;
    xch[h * 128 + r] = l;
    bar_sync(pair_bar, kRowGroupThreads);
    float l_row = xch[r];
#pragma unroll
    for (int g = 1; g < NG; ++g) l_row += xch[g * 128 + r];
    const uint32_t t_last = tile_ctr - 1;  // its commit covers every earlier MMA too
    ok = wait(bar(Ly::B_ODONE + static_cast<int>(t_last & 1u)), (t_last >> 1) & 1u, kSiteODone);
    ok = __all_sync(0xFFFFFFFFu, ok);
    if (!ok) {
      *pair_fail = 1;  // no pair barrier remains in this unit; the next vote settles it
      continue;
    }
    tc_fence_after();
    store_row<HD, OCOLS>(p, U, tok, head, h * OCOLS, lane_tmem + h * OCOLS, m, l_row, h == 0);
    tc_fence_before();
  }
}

// ------------------------------------------ softmax, HD = 128: whole rows
// The two softmax warpgroups take alternate K/V tiles of a unit: warpgroup b
// (warps 4b .. 4b+3, warp w reading TMEM lanes 32 (w % 4) ..) takes the tiles
// whose CTA-wide index t has t % 2 == b, whole rows of them (128 logits per
// thread), and keeps its own online softmax (m_b, l_b) and its own O_b in
// TMEM, into which the MMA warp accumulates P_t V_t.  The two partial
// softmaxes of a row are merged exactly at the unit's epilogue:
//   m = max(m_0, m_1),  w_b = 2^(m_b - m),
//   O = (w_0 O_0 + w_1 O_1) / (w_0 l_0 + w_1 l_1)
// -- the same single softmax over all the unit's keys (a split of the sum,
// not a second launch: both halves live in one CTA's TMEM).  No per-tile
// exchange between warps is needed, each thread's per-tile work is spread
// over twice the logits, and two tiles are in the softmax stage at once.
// The row group (warps w and w + 4, one named barrier) meets only at the
// epilogue.
//
// Ordering.  Warpgroup b observes every completion of S_FULL[b] (its
// tiles).  Tile t - 2's P.V, the previous product into O_b, is complete by
// then: one thread issues every MMA, QK^T of tile t after that P.V, and a
// commit arrives only once all of the thread's earlier MMAs are complete.
// So O_b may be rescaled during tile t without a wait on O_DONE[b]; P.V of
// tile t is issued after its P arrival, so no product into O_b is in flight
// during the rescale.  O_DONE[b] is waited for only at the epilogue, for the
// warpgroup's last P.V of the unit: every earlier phase of it is complete
// then, so the parity wait is never more than one phase behind.  The row
// group then meets, and meets again once both have read O_0 and O_1, before
// either can arrive for the next unit's first tile (whose P.V overwrites an
// O).
template <bool SPLIT, bool PAIR2, int VF16, int CL>
__device__ __forceinline__ void softmax_role_rows(const PrefillParams& p, uint32_t sbase,
                                                  uint32_t tmem, const BoundedWait& wait) {
  constexpr int HD = 128;
  using Ly = Layout<HD>;
  static_assert(Ly::SPLIT_O && kColGroups == 2, "two warpgroups, two O accumulators");
  auto bar = [&](int i) { return sbase + Ly::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  constexpr int CH = kBKV / 32;  // 32-column TMEM loads per row
  const int warp = threadIdx.x >> 5;
  const uint32_t b = static_cast<uint32_t>(warp >> 2);   // tile parity and O buffer
  const int r = ((warp & 3) << 5) | (threadIdx.x & 31);  // row == TMEM lane
  const uint32_t pair_bar = 1u + static_cast<uint32_t>(warp & 3);
  const uint32_t lane_tmem = tmem + (static_cast<uint32_t>(r & ~31) << 16);
  const uint32_t s_tmem = lane_tmem + HD + b * kBKV;
  float* xch = reinterpret_cast<float*>(__cvta_shared_to_generic(sbase + Ly::OFF_XCH));
  volatile int* pair_fail = reinterpret_cast<volatile int*>(
      __cvta_shared_to_generic(sbase + Ly::OFF_PFAIL)) + (warp & 3);
  const float sl2 = p.scale_log2;
  uint32_t tile_ctr = 0;  // CTA-wide tile index (the MMA warp's sequence)
  bool drop_one = (p.debug_flags & kDebugDropArrive) && blockIdx.x == 0 && threadIdx.x == 0;

  for (int ur = 0, u = unit_of<CL>(0); u < p.num_units; u = unit_of<CL>(++ur)) {
    const Unit U = decode_unit(p, u);
    const int tok = U.q0 + (p.packed ? r / p.group : r);
    const int head = p.packed ? U.h + r % p.group : U.h;
    CacheWalk walk;
    walk.init(U.L, p.P, p.S);
    walk.skip(U.v0 < U.n_cache ? U.v0 : U.n_cache);
    float m = -INFINITY;  // this warpgroup's reference max (log2 units), per row
    float l = 0.f;        // its running sum of 2^(x - m)
    int mine = 0;         // tiles of this unit this warpgroup took
    uint32_t t_mine = 0;  // the last of them
    bool ok = true;

    for (int v = 0; v < U.n_tiles; ++v) {
      const uint32_t t = tile_ctr + static_cast<uint32_t>(v);
      const int va = U.v0 + v;
      const bool in_cache = va < U.n_cache;
      // The walk advances over every cache tile, also the other warpgroup's.
      const int tile = in_cache ? walk.next() : 0;
      if ((t & 1u) != b || !ok) continue;
      uint32_t mw[4];
      if (in_cache) {
        if (walk.last_full) {
          mw[0] = mw[1] = mw[2] = mw[3] = 0xFFFFFFFFu;
        } else {
          walk.column_mask(tile, mw);
        }
      } else {
        const int lim0 = tok - kBKV * (va - U.n_cache) + 1;
        const int lim = lim0 < 0 ? 0 : (lim0 > kBKV ? kBKV : lim0);
#pragma unroll
        for (int q = 0; q < 4; ++q) mw[q] = causal_word(lim, q);
      }
      const bool need_mask =
          __any_sync(0xFFFFFFFFu, (mw[0] & mw[1] & mw[2] & mw[3]) != 0xFFFFFFFFu);
      ok = __all_sync(0xFFFFFFFFu, wait(bar(Ly::B_SFULL + b), (t >> 1) & 1u, kSiteSFull));
      if (!ok) {
        *pair_fail = 1;  // settled at the epilogue barrier
        continue;
      }
      tc_fence_after();

      // Pass 1: the row's 128 logits (all TMEM loads in flight together),
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

      // Lazy rescale: the reference moves only when the row's new logits
      // exceed it by more than 2^8 (the final O / l is the same either way).
      const float m_new = fmaxf(m, m_tile);
      const bool need = mine > 0 && m_new > m + 8.f;
      const float alpha = need ? ex2_approx(m - m_new) : 1.f;
      if (mine == 0 || need) m = m_new;

      // Pass 2: p = 2^(x - m), its row sum, and P over the tile's S columns.
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

      // A row whose reference moved scales its O_b in place: every product
      // into O_b so far (up to tile t - 2) is complete (S_FULL of tile t was
      // committed after it), and P.V of tile t waits for this warpgroup's
      // arrival below.
      if (__any_sync(0xFFFFFFFFu, need)) {
        const uint32_t o_tmem = lane_tmem + (b ? Ly::O_COL1 : 0u);
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
      if (PAIR2) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) {
          if (drop_one) {
            drop_one = false;  // fault-injection hook: this arrival never happens
          } else {
            count_arrive(p.bar_counts, 1u, Ly::B_PFULL + static_cast<int>(b), 1);
            mbar_arrive_remote(mapa_shared(bar(Ly::B_PFULL + static_cast<int>(b)), 0));
          }
        }
      } else if (drop_one) {
        drop_one = false;  // fault-injection hook: this arrival never happens
      } else {
        count_arrive(p.bar_counts, 1u, Ly::B_PFULL + static_cast<int>(b), 1);
        mbar_arrive(bar(Ly::B_PFULL + static_cast<int>(b)));
      }
      ++mine;
      t_mine = t;
    }
    tile_ctr += static_cast<uint32_t>(U.n_tiles);

    // Epilogue.  Each warpgroup waits for its own last P.V on its O_DONE
    // (the only phase of it that can still be open), posts (m_b, l_b), and
    // the row group meets.
    if (ok && mine > 0) {
      ok = __all_sync(0xFFFFFFFFu,
                      wait(bar(Ly::B_ODONE + b), (t_mine >> 1) & 1u, kSiteODone));
      if (!ok) *pair_fail = 1;
    }
    xch[(2 * b) * 128 + r] = mine > 0 ? m : -INFINITY;
    xch[(2 * b + 1) * 128 + r] = l;
    tc_fence_before();
    bar_sync(pair_bar, kRowGroupThreads);
    if (*pair_fail) break;  // read by both warps after the same barrier
    tc_fence_after();
    const float m0 = xch[r], l0 = xch[128 + r];
    const float m1 = xch[256 + r], l1 = xch[384 + r];
    const float mm = fmaxf(m0, m1);
    const float w0 = m0 == -INFINITY ? 0.f : ex2_approx(m0 - mm);
    const float w1 = m1 == -INFINITY ? 0.f : ex2_approx(m1 - mm);
    const float l_row = w0 * l0 + w1 * l1;
    // Which O buffers hold this unit's products (a one-tile unit has none in
    // O_1, whose contents are then stale): uniform over the unit.
    const bool has0 = U.n_tiles > 0 && (((tile_ctr - U.n_tiles) & 1u) == 0 || U.n_tiles > 1);
    const bool has1 = U.n_tiles > 0 && (((tile_ctr - U.n_tiles) & 1u) == 1 || U.n_tiles > 1);
    store_row_merged<HD, HD / 2>(p, U, tok, head, static_cast<int>(b) * (HD / 2),
                                 lane_tmem + b * (HD / 2), lane_tmem + Ly::O_COL1 + b * (HD / 2),
                                 has0 ? w0 : 0.f, has1 ? w1 : 0.f, has0, has1, mm, l_row, b == 0);
    // Both warps are done reading O_0 and O_1 before either arrives for the
    // next unit's first tile.
    tc_fence_before();
    bar_sync(pair_bar, kRowGroupThreads);
  }
}

// ------------------------------------------------------------------ kernel
template <int HD, bool SPLIT, int VF16>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
  using Ly = Layout<HD>;
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
      mbar_init(bar(i), (i == Ly::B_PFULL || i == Ly::B_PFULL + 1) ? Ly::P_THREADS : 1u);
    *abort_flag = 0;
    for (int i = 0; i < 4; ++i) reinterpret_cast<volatile int*>(smem + Ly::OFF_PFAIL)[i] = 0;
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
    if constexpr (Ly::SPLIT_O) {
      reg_alloc_inc<kSoftmaxRegs>();
      softmax_role_rows<SPLIT, false, VF16, 1>(p, sbase, tmem, wait);
    } else {
      softmax_role<HD, SPLIT, false, VF16, 1>(p, sbase, tmem, wait);
    }
  } else {
    if constexpr (Ly::SPLIT_O) reg_alloc_dec<kOtherRegs>();
    if (warp == kProducerWarp) {
      if (lane == 0) {
        // The staged fp16 V is written by the kernel this one depends on.
        if constexpr (VF16 == kVF16All) griddep_wait();
        producer_role<HD>(p, sbase, wait);
      }
    } else if (warp == kWriterWarp) {
      if (p.k_cache_w != nullptr) kv_write_lanes<HD, VF16 != kVBf16, 1>(p, lane);
    } else if (warp == kMmaWarp) {
      mma_role<HD, SPLIT, VF16>(p, sbase, tmem, wait);
    }
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
