// Host-side work plan of one prefill launch.
//
// A row block is (sequence b, 128-row q block qb); its unit (one q head)
// walks the virtual tile index v over n_cache cache tiles then the causal
// current tiles 0..qb.  The plan lists work blocks, each a row block with a
// slice [v0, v1) of that walk, longest first (a persistent grid takes them in
// order, so the longest start first).
//
// Split-KV (for small chunks and decode): when a few long walks would leave
// most SMs idle, a row block's walk is cut into pieces (their length chosen
// by a cost model of the grid's rounds, below).  Each piece writes fp32 O / l and its LSE for the block's
// valid rows into a workspace ("partial rows"), and a merge pass combines
// the pieces of each row by their LSE.  This is the single-GPU counterpart of
// the pages' spilled running (m, l, acc) for very long contexts (PCP
// ring-cache PR, Design section), with the walk cut across SMs instead of
// across launches.
#pragma once

#include <algorithm>
#include <string>
#include <vector>

#include "cpattn.h"
#include "merge.cuh"
#include "walk.cuh"

namespace cpattn {

enum : int { kRegionAll = 0, kRegionCache = 1, kRegionCurrent = 2 };
constexpr int kSplitOff = -1;   // never split
constexpr int kSplitAuto = 0;   // split when the cost model says it pays
// Shortest piece the automatic policy considers.  16 kept a 37-row chunk
// against 15000 cached tokens at 35 pieces (49 us); 8 lets it take 70, and
// pieces of 8 tiles measured 42 us.
constexpr int kMinPieceTiles = 8;
constexpr int kUnitOverheadTiles = 2;  // pipeline fill and drain of one unit, in tile times
constexpr int kMaxPieceCandidates = 64;
// Costs of a piece beyond its tiles, in tile times (a tile takes ~1.5 us per
// SM or SM pair): writing its fp32 partial rows (~64 KB per SM per tile
// time), and the merge pass reading all partials back (~10 MB GPU-wide per
// tile time).  Measured: without them the model cut 128-row blocks into
// pieces that then ran 5 % slower than the fused walk.
constexpr long long kPieceWriteBytesPerTile = 64 << 10;
constexpr long long kMergeBytesPerTile = 10 << 20;

// Cost model of a plan: the persistent grid deals units out in rounds of E
// in list order, and a unit costs its tiles plus a fixed fill/drain
// overhead.  `lens` holds one entry per work block, longest first (any
// per-unit extra cost already added); each block has units_per_block units.
// The kernels deal each round in snake order (executor e takes slot e of
// even rounds, slot E-1-e of odd ones); the model charges every round its
// first, longest unit -- the load of executor 0 under a cyclic deal -- which
// bounds every executor's snake load from above: O(rounds), no per-executor
// state.
inline long long cyclic_makespan(const std::vector<int>& lens, int units_per_block,
                                 int executors) {
  const long long total = static_cast<long long>(lens.size()) * units_per_block;
  const long long E = std::max(executors, 1);
  long long m = 0;
  for (long long i = 0; i < total; i += E) m += lens[static_cast<size_t>(i / units_per_block)] + kUnitOverheadTiles;
  return m;
}
constexpr int kMaxVirtualTiles = 65535;  // v0 and v1 are packed in 16 bits each

// Makespan of units dealt to E executors in snake order (executor e takes
// slot e of even rounds, slot E-1-e of odd ones), each costing its tiles plus
// the fill/drain overhead; lens[u] is unit u's tiles, in unit-index order.
inline long long snake_makespan(const std::vector<int>& lens, int executors) {
  const int E = std::max(executors, 1);
  std::vector<long long> load(static_cast<size_t>(E), 0);
  for (size_t u = 0; u < lens.size(); ++u) {
    const long long r = static_cast<long long>(u) / E;
    const int slot = static_cast<int>(u % E);
    load[static_cast<size_t>((r & 1) ? E - 1 - slot : slot)] += lens[u] + kUnitOverheadTiles;
  }
  return *std::max_element(load.begin(), load.end());
}

// Whether to deal units kv-head-major (see PrefillParams::kv_major): units
// that run at once then read one kv head's K/V, so it is fetched from DRAM
// about once instead of once per round of the grid.  Taken when it costs the
// grid at most 1 % of the longest-first order's makespan (the measure of a
// compute-bound launch); block_lens: the work blocks' tiles, longest first;
// per_kv: units of one kv head per block.
inline bool prefer_kv_major(const std::vector<int>& block_lens, int per_kv, int nkv,
                            int executors) {
  const size_t units = block_lens.size() * static_cast<size_t>(per_kv) * nkv;
  if (nkv < 2 || units <= static_cast<size_t>(executors)) return false;
  std::vector<int> lf, kv;
  lf.reserve(units);
  kv.reserve(units);
  for (int len : block_lens)
    for (int j = 0; j < per_kv * nkv; ++j) lf.push_back(len);
  for (int g = 0; g < nkv; ++g)
    for (int len : block_lens)
      for (int j = 0; j < per_kv; ++j) kv.push_back(len);
  return snake_makespan(kv, executors) * 100 <= snake_makespan(lf, executors) * 101;
}

// A work block entry of the kernel's table: sequence b (< 128), first unit
// head hoff (< 16384), q block qb (< 2048: a launch has at most
// CPATTN_MAX_ROW_BLOCKS row blocks).
inline uint32_t pack_block(int b, int qb, int hoff) {
  return (static_cast<uint32_t>(b) << 25) | (static_cast<uint32_t>(hoff) << 11) |
         static_cast<uint32_t>(qb);
}
static_assert(CPATTN_MAX_SEQS <= 128 && CPATTN_MAX_ROW_BLOCKS <= 2048, "work block entry bits");

struct WorkBlock {
  int b, qb, v0, v1;
  int part;  // -1: writes the output; else the first partial row of a piece
};

struct SplitGroup {
  int b, q0, rows, n, part0;  // piece s has partial rows part0 + s * rows ..
};

struct WorkPlan {
  std::vector<int> ncache;         // cache tiles per sequence
  std::vector<WorkBlock> blocks;   // longest first
  std::vector<SplitGroup> groups;  // row blocks cut into pieces
  long long partial_rows = 0;
};

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace bytes of a plan: fp32 O / l then the LSE, both 256-byte aligned.
inline size_t plan_workspace_bytes(const WorkPlan& w, int nq, int hd) {
  if (w.partial_rows == 0) return 0;
  const size_t rows = static_cast<size_t>(w.partial_rows) * static_cast<size_t>(nq);
  return align256(rows * static_cast<size_t>(hd) * 4) + align256(rows * 4);
}

// region: kRegionAll, or the two-launch variant's cache-only / current-only
// halves (never split).  split: kSplitOff, kSplitAuto, or > 0 = cut every walk
// longer than that many tiles into pieces of at most that many.  executors:
// how many units run at once (SMs, or SM pairs); units_per_block: units one
// work block gives them (q heads, or q-head pairs).  Returns false with `why`
// when the plan exceeds the kernel's tables.
inline bool make_plan(const cpattn_config& c, int num_seqs, const int32_t* cache_lens,
                      const int32_t* chunk_lens, int region, int split, int executors,
                      int units_per_block, int block_tokens, WorkPlan* plan, std::string* why) {
  plan->ncache.assign(num_seqs, 0);
  plan->blocks.clear();
  plan->groups.clear();
  plan->partial_rows = 0;
  struct Row { int b, qb, v0, v1, rows; };
  std::vector<Row> rows;
  for (int b = 0; b < num_seqs; ++b) {
    const int nc = cache_tile_count(cache_lens[b], c.num_shards, c.shard_capacity);
    plan->ncache[b] = nc;
    if (region == kRegionCache && nc == 0) continue;  // no cache-only work
    // Row blocks of block_tokens chunk tokens (128, or 128 / G when packed);
    // a block's walk ends with the current tile of its last token.
    const int nqb = (chunk_lens[b] + block_tokens - 1) / block_tokens;
    for (int qb = 0; qb < nqb; ++qb) {
      const int last = std::min((qb + 1) * block_tokens, static_cast<int>(chunk_lens[b])) - 1;
      const int v0 = region == kRegionCurrent ? nc : 0;
      const int v1 = region == kRegionCache ? nc : nc + last / kBKV + 1;
      if (v1 > kMaxVirtualTiles) {
        *why = "a cache walk longer than 65535 - q blocks tiles";
        return false;
      }
      rows.push_back({b, qb, v0, v1, std::min(block_tokens, chunk_lens[b] - qb * block_tokens)});
    }
  }

  // Which row blocks to cut, and into how many pieces.  Pieces of at most
  // `target` tiles; the automatic policy tries the targets ceil(n_max / k) and
  // keeps the one whose modelled makespan is lowest, if it beats the unsplit
  // plan by 10 %.
  std::vector<int> pieces(rows.size(), 1);
  std::vector<int> order(rows.size());  // row blocks, longest walk first
  for (size_t i = 0; i < rows.size(); ++i) order[i] = static_cast<int>(i);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
    return rows[a].v1 - rows[a].v0 > rows[b].v1 - rows[b].v0;
  });
  auto cut = [&](int target, std::vector<int>* out) {
    out->assign(rows.size(), 1);
    size_t nblocks = rows.size();
    int groups = 0;
    for (int i : order) {
      const int n = rows[i].v1 - rows[i].v0;
      if (n <= target) break;
      const int k = (n + target - 1) / target;
      if (groups == kMaxSplitGroups || nblocks + k - 1 > CPATTN_MAX_ROW_BLOCKS) break;
      (*out)[i] = k;
      nblocks += k - 1;
      ++groups;
    }
  };
  const int heads_per_unit = c.num_q_heads / std::max(units_per_block, 1);
  std::vector<int> lens;
  lens.reserve(rows.size() * 4);
  auto makespan = [&](const std::vector<int>& k) {
    lens.clear();
    long long merge_bytes = 0;
    for (size_t i = 0; i < rows.size(); ++i) {
      const int n = rows[i].v1 - rows[i].v0;
      // A piece also writes rows x heads x HD fp32 partials.
      const long long wbytes =
          static_cast<long long>(rows[i].rows) * heads_per_unit * c.head_dim * 4;
      const int extra = k[i] > 1 ? static_cast<int>((wbytes + kPieceWriteBytesPerTile - 1) /
                                                    kPieceWriteBytesPerTile)
                                 : 0;
      if (k[i] > 1)
        merge_bytes += static_cast<long long>(k[i]) * rows[i].rows * c.num_q_heads *
                       (c.head_dim + 1) * 4;
      for (int s = 0; s < k[i]; ++s)
        lens.push_back(static_cast<int>(static_cast<long long>(n) * (s + 1) / k[i] -
                                        static_cast<long long>(n) * s / k[i]) + extra);
    }
    std::sort(lens.begin(), lens.end(), [](int a, int b) { return a > b; });
    return cyclic_makespan(lens, units_per_block, executors) +
           (merge_bytes + kMergeBytesPerTile - 1) / kMergeBytesPerTile;
  };
  if (split != kSplitOff && region == kRegionAll && !rows.empty()) {
    if (split > 0) {
      cut(split, &pieces);
    } else {
      int n_max = 0;
      long long total = 0;
      for (const Row& r : rows) {
        n_max = std::max(n_max, r.v1 - r.v0);
        total += static_cast<long long>(units_per_block) * (r.v1 - r.v0 + kUnitOverheadTiles);
      }
      const long long ideal = (total + executors - 1) / std::max(executors, 1);
      const long long base = makespan(pieces);
      if (base * 10 > ideal * 11) {  // rounds of the grid leave more than 10 % idle
        long long best = base;
        std::vector<int> trial;
        // k = 2..8, then a geometric ladder to 64: the makespan moves in
        // steps of whole grid rounds, so finer k rarely matters.
        static const int kLadder[] = {2, 3, 4, 5, 6, 7, 8, 10, 12, 14, 16, 20, 24, 28, 32,
                                      40, 48, 56, 64};
        for (int k : kLadder) {
          if (k > kMaxPieceCandidates) break;
          const int target = (n_max + k - 1) / k;
          if (target < kMinPieceTiles) break;
          cut(target, &trial);
          const long long m = makespan(trial);
          if (m < best) {
            best = m;
            pieces = trial;
          }
        }
        if (best * 10 > base * 9) pieces.assign(rows.size(), 1);  // under 10 %: not worth it
      }
    }
  }

  for (size_t i = 0; i < rows.size(); ++i) {
    const Row& r = rows[i];
    const int k = pieces[i];
    if (k == 1) {
      plan->blocks.push_back({r.b, r.qb, r.v0, r.v1, -1});
      continue;
    }
    const int n = r.v1 - r.v0;
    const int part0 = static_cast<int>(plan->partial_rows);
    plan->groups.push_back({r.b, r.qb * block_tokens, r.rows, k, part0});
    for (int s = 0; s < k; ++s) {
      const int a = r.v0 + static_cast<int>(static_cast<long long>(n) * s / k);
      const int e = r.v0 + static_cast<int>(static_cast<long long>(n) * (s + 1) / k);
      plan->blocks.push_back({r.b, r.qb, a, e, part0 + s * r.rows});
    }
    plan->partial_rows += static_cast<long long>(k) * r.rows;
  }
  if (plan->blocks.size() > CPATTN_MAX_ROW_BLOCKS) {
    *why = "more than CPATTN_MAX_ROW_BLOCKS row blocks";
    return false;
  }
  if (plan->partial_rows * c.num_q_heads >= (1LL << 31)) {
    *why = "split-KV partial rows exceed the 32-bit index range";
    return false;
  }
  std::stable_sort(plan->blocks.begin(), plan->blocks.end(),
                   [](const WorkBlock& a, const WorkBlock& b) { return a.v1 - a.v0 > b.v1 - b.v0; });
  return true;
}

}  // namespace cpattn
