// C-ABI library: argument checks, tensor-map encoding, launches.
// Declarations and contracts: include/cpattn.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "cpattn.h"
#include "prefill.cuh"
#include "prefill_pair.cuh"
#include "prefill_pingpong.cuh"
#include "walk.cuh"
#include "write_kv.cuh"
#include "merge.cuh"
#include "plan.h"

static_assert(cpattn::kCountRecord == CPATTN_COUNT_RECORD && cpattn::kCountBars == CPATTN_COUNT_BARS,
              "barrier-count record layout");
static_assert(cpattn::Layout<128>::NBAR <= cpattn::kCountBars &&
                  cpattn::Layout<256>::NBAR <= cpattn::kCountBars &&
                  cpattn::PingPongLayout::NBAR <= cpattn::kCountBars,
              "every barrier has a count slot");

struct cpattn_ctx {
  cpattn_config cfg;
  int device = -1;
  int num_sms = 0;
  int* d_status = nullptr;           // device status word (timeouts)
  // [HD == 256][split P][pairing mode][V form: kVBf16, kVF16Cache, kVF16All]: 0 until set up
  int grid_cap[2][2][4][3] = {};
  // Head pairing for even group sizes (cpattn_config.pairing, or the
  // CPATTN_PAIRING override): 2 = 2-SM MMA pairs, 3 = two query tiles per CTA
  // (HD = 128; 2 at HD = 256), 0 = off.
  int pair_mode = 2;
  // Split-KV: a caller-owned device workspace and the policy (kSplitOff,
  // kSplitAuto, or a forced piece length in tiles); off until registered.
  void* split_ws = nullptr;
  size_t split_ws_bytes = 0;
  // fp16 V cache: a caller-owned device buffer where the prefill entry
  // points stage the chunk's V in fp16 (cpattn_set_v_staging); none: the
  // chunk's tiles take the bf16 hi+lo P pair against bf16 V_new.
  void* v_stage = nullptr;
  size_t v_stage_bytes = 0;
  int split_policy = cpattn::kSplitOff;
  // GQA packing for short-chunk launches (cpattn_config.gqa_packing, or the
  // CPATTN_GQA_PACKING override).
  bool gqa_packing = true;
  std::vector<int> block_lens;  // scratch of the unit-order choice
  // Unit order (test override CPATTN_UNIT_ORDER): 0 chosen by the cost
  // model, 1 longest first, 2 kv-head-major.
  int unit_order = 0;
  // Barrier-count build: caller-owned per-CTA count records, and their bytes.
  uint32_t* bar_counts = nullptr;
  size_t bar_counts_bytes = 0;
  int debug_flags = 0;
  unsigned long long timeout_ns = 1000ull * 1000 * 1000;
  bool debug_sync = false;
  std::string last_error;
};

namespace {

using cpattn::kBKV;
using cpattn::kBQ;

cpattn_status fail(cpattn_ctx* ctx, cpattn_status s, const std::string& msg) {
  if (ctx != nullptr) ctx->last_error = msg;
  return s;
}

cpattn_status cuda_fail(cpattn_ctx* ctx, cudaError_t e, const char* what) {
  return fail(ctx, CPATTN_E_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 3-D bf16 tensor map with 128-byte swizzle: dims (d0 innermost), byte
// strides of dims 1 and 2, box (b0, b1, b2).
bool encode3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t st1, uint64_t st2, uint32_t b0, uint32_t b1, uint32_t b2) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {st1, st2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Checks shared by write_kv and prefill.
cpattn_status check_seqs(cpattn_ctx* ctx, int32_t num_seqs, const int32_t* cache_lens,
                         const int32_t* chunk_lens) {
  if (num_seqs < 1) return fail(ctx, CPATTN_E_INVALID, "num_seqs must be >= 1");
  if (num_seqs > CPATTN_MAX_SEQS)
    return fail(ctx, CPATTN_E_UNSUPPORTED,
                "num_seqs " + std::to_string(num_seqs) + " exceeds CPATTN_MAX_SEQS");
  if (cache_lens == nullptr || chunk_lens == nullptr)
    return fail(ctx, CPATTN_E_INVALID, "cache_lens / chunk_lens must not be NULL");
  const cpattn_config& c = ctx->cfg;
  const long long cap = static_cast<long long>(c.num_shards) * c.shard_capacity;
  for (int b = 0; b < num_seqs; ++b) {
    if (cache_lens[b] < 0)
      return fail(ctx, CPATTN_E_INVALID, "cache_lens[" + std::to_string(b) + "] < 0");
    if (chunk_lens[b] < 0 || chunk_lens[b] > c.chunk_size)
      return fail(ctx, CPATTN_E_INVALID,
                  "chunk_lens[" + std::to_string(b) + "] outside [0, chunk_size]");
    if (static_cast<long long>(cache_lens[b]) + chunk_lens[b] > cap)
      return fail(ctx, CPATTN_E_INVALID,
                  "sequence " + std::to_string(b) + ": cache_len + chunk_len exceeds P*S");
  }
  const long long cache_rows =
      static_cast<long long>(num_seqs) * c.num_kv_heads * c.num_shards * c.shard_capacity;
  const long long tokens = static_cast<long long>(num_seqs) * c.chunk_size;
  if (cache_rows + kBKV >= (1LL << 31) || tokens + kBQ >= (1LL << 31))
    return fail(ctx, CPATTN_E_UNSUPPORTED, "cache or token row count exceeds 2^31");
  return CPATTN_OK;
}

cpattn_status after_launch(cpattn_ctx* ctx, cudaStream_t stream, const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(ctx, e, what);
  if (ctx->debug_sync) return cpattn_sync_status(ctx, stream);
  return CPATTN_OK;
}

// The HD = 128 kernels move registers between warpgroups (setmaxnreg): the
// two softmax warpgroups' increase waits until the third warpgroup's
// decrease has freed enough of the CTA's launch-sized pool, which holds
// exactly enough only if the kernel was compiled to kLaunchRegs registers
// per thread.  A kernel built otherwise is never launched.
bool register_split_ok(const void* kernel) {
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return fa.numRegs == cpattn::kLaunchRegs && fa.maxThreadsPerBlock >= cpattn::kThreads;
}

template <int HD, bool SPLIT, int MODE, int VF16>
cpattn_status launch_prefill(cpattn_ctx* ctx, cpattn::PrefillParams* prm, cudaStream_t stream) {
  static_assert(MODE == 0 || MODE == 2 || (MODE == 3 && HD == 128),
                "pairing modes: 0 (none), 2 (2-SM MMA pairs), 3 (two query tiles, HD = 128)");
  constexpr bool MC = MODE == 2;  // launched as clusters of two CTAs
  constexpr int SMEM_BYTES =
      MODE == 3 ? cpattn::PingPongLayout::SMEM_BYTES : cpattn::Layout<HD>::SMEM_BYTES;
  void (*kernel)(cpattn::PrefillParams);
  if constexpr (MODE == 3)
    kernel = cpattn::prefill_kernel_pingpong<SPLIT, VF16>;
  else if constexpr (MODE == 2)
    kernel = cpattn::prefill_kernel_pair2<HD, SPLIT, VF16>;
  else
    kernel = cpattn::prefill_kernel<HD, SPLIT, VF16>;
  int& grid_cap = ctx->grid_cap[HD == 256][SPLIT][MODE][VF16];
  if (grid_cap == 0) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaFuncSetAttribute(prefill)");
    if (MODE != 3 && cpattn::Layout<HD>::SPLIT_O &&
        !register_split_ok(reinterpret_cast<const void*>(kernel)))
      return fail(ctx, CPATTN_E_UNSUPPORTED,
                  "the HD = 128 prefill kernel was not built with the registers per thread "
                  "its warpgroup register split assumes");
    grid_cap = ctx->num_sms;
    if (MC) {
      // Persistent grid of co-resident CTA pairs.
      cudaLaunchConfig_t q = {};
      q.gridDim = dim3(2 * ctx->num_sms, 1, 1);
      q.blockDim = dim3(cpattn::kThreads, 1, 1);
      q.dynamicSmemBytes = SMEM_BYTES;
      cudaLaunchAttribute a[1];
      a[0].id = cudaLaunchAttributeClusterDimension;
      a[0].val.clusterDim.x = 2;
      a[0].val.clusterDim.y = 1;
      a[0].val.clusterDim.z = 1;
      q.attrs = a;
      q.numAttrs = 1;
      int clusters = 0;
      e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &q);
      if (e != cudaSuccess || clusters < 1) {
        cudaGetLastError();
        return fail(ctx, CPATTN_E_CUDA, "no co-resident CTA pair for the paired prefill kernel");
      }
      grid_cap = std::min(2 * clusters, ctx->num_sms & ~1);
    }
  }
  // A CTA of MODE 3 takes two units (a head pair) per round.
  int grid = std::min(MODE == 3 ? prm->num_units / 2 : prm->num_units, grid_cap);
  if (MC) grid &= ~1;
  if (ctx->bar_counts != nullptr) {
    if (ctx->bar_counts_bytes < static_cast<size_t>(grid) * cpattn::kCountRecord * 4)
      return fail(ctx, CPATTN_E_INVALID,
                  "the barrier-count buffer holds fewer records than the launch's " +
                      std::to_string(grid) + " CTAs");
    prm->bar_counts = ctx->bar_counts;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(cpattn::kThreads, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = MC ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if constexpr (VF16 == cpattn::kVF16All) {
    // A programmatic dependent of the V staging kernel just launched on the
    // stream: its prologue overlaps the staging, and its producer waits for
    // the staging grid (griddep_wait) before the first copy.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, *prm);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "prefill launch");
  return after_launch(ctx, stream, "prefill launch");
}

// The pairing mode a launch runs in: none for packed units (they hold a
// whole kv group already) or odd group sizes; two query tiles per CTA only
// at HD = 128 (the 2-SM pairs at HD = 256, whose O fills half of TMEM).
int launch_pair_mode(const cpattn_ctx* ctx, bool packed) {
  const cpattn_config& c = ctx->cfg;
  if (packed || (c.num_q_heads / c.num_kv_heads) % 2 != 0) return 0;
  if (ctx->pair_mode == 3 && c.head_dim != 128) return 2;
  return ctx->pair_mode;
}

// The plan's executors and units per work block: SM pairs and q-head pairs
// for CTA pairs, SMs and q-head pairs for two query tiles per CTA, else SMs
// and q heads (148 SMs when no device is present, for host-side planning).
void plan_shape(const cpattn_ctx* ctx, bool packed, int* executors, int* units_per_block) {
  const int sms = ctx->num_sms > 0 ? ctx->num_sms : 148;
  if (packed) {  // one unit per kv head, unpaired
    *executors = sms;
    *units_per_block = ctx->cfg.num_kv_heads;
    return;
  }
  const int mode = launch_pair_mode(ctx, packed);
  *executors = mode == 2 ? sms / 2 : sms;
  *units_per_block = mode != 0 ? ctx->cfg.num_q_heads / 2 : ctx->cfg.num_q_heads;
}

// GQA packing: a unit's 128 rows become (token, q head of one kv group) when
// every chunk is short (<= 64 tokens) and the group size G is a power of two
// in [2, 128], so a decode step fills 128 / G tokens x G heads instead of 1
// row of 128.  Returns the tokens per row block (128 when not packed).
constexpr int kPackMaxTokens = 64;
int pack_block_tokens(const cpattn_ctx* ctx, int32_t num_seqs, const int32_t* chunk_lens,
                      int region) {
  const int G = ctx->cfg.num_q_heads / ctx->cfg.num_kv_heads;
  if (!ctx->gqa_packing || region != cpattn::kRegionAll || G < 2 || G > kBQ || (G & (G - 1)) != 0)
    return kBQ;
  for (int b = 0; b < num_seqs; ++b)
    if (chunk_lens[b] > kPackMaxTokens) return kBQ;
  return kBQ / G;
}

template <int HD, int VF16>
cpattn_status dispatch_prefill_hd(cpattn_ctx* ctx, cpattn::PrefillParams* prm, cudaStream_t st,
                                  bool split, int mode) {
  if constexpr (VF16 == cpattn::kVF16All) {
    // Every tile takes one fp16 product: the form has no fast_p variant.
    if constexpr (HD == 128) {
      if (mode == 3) return launch_prefill<HD, true, 3, VF16>(ctx, prm, st);
    }
    if (mode == 2) return launch_prefill<HD, true, 2, VF16>(ctx, prm, st);
    return launch_prefill<HD, true, 0, VF16>(ctx, prm, st);
  } else {
    if constexpr (HD == 128) {
      if (mode == 3) return split ? launch_prefill<HD, true, 3, VF16>(ctx, prm, st)
                                  : launch_prefill<HD, false, 3, VF16>(ctx, prm, st);
    }
    if (mode == 2) return split ? launch_prefill<HD, true, 2, VF16>(ctx, prm, st)
                                : launch_prefill<HD, false, 2, VF16>(ctx, prm, st);
    return split ? launch_prefill<HD, true, 0, VF16>(ctx, prm, st)
                 : launch_prefill<HD, false, 0, VF16>(ctx, prm, st);
  }
}

// The V form of a launch: a bf16 V cache; an fp16 one with the chunk's V as
// bf16 V_new; or with the chunk's V staged in fp16 (every tile one fp16
// product, so the form needs no fast_p variant: it runs as the SPLIT one).
cpattn_status dispatch_prefill(cpattn_ctx* ctx, cpattn::PrefillParams* prm, cudaStream_t st,
                               bool packed, bool v_staged) {
  const int HD = ctx->cfg.head_dim;
  const bool split = ctx->cfg.fast_p == 0 || v_staged;
  const bool vf16 = ctx->cfg.v_cache_f16 != 0;
  // Pair adjacent q heads of one kv head when the group size allows.
  const int mode = launch_pair_mode(ctx, packed);
  if (HD == 256) {
    if (v_staged) return dispatch_prefill_hd<256, cpattn::kVF16All>(ctx, prm, st, split, mode);
    return vf16 ? dispatch_prefill_hd<256, cpattn::kVF16Cache>(ctx, prm, st, split, mode)
                : dispatch_prefill_hd<256, cpattn::kVBf16>(ctx, prm, st, split, mode);
  }
  if (v_staged) return dispatch_prefill_hd<128, cpattn::kVF16All>(ctx, prm, st, split, mode);
  return vf16 ? dispatch_prefill_hd<128, cpattn::kVF16Cache>(ctx, prm, st, split, mode)
              : dispatch_prefill_hd<128, cpattn::kVBf16>(ctx, prm, st, split, mode);
}

// Combine the split-KV pieces of every split row block into the output.
cpattn_status launch_splitkv_merge(cpattn_ctx* ctx, const cpattn::WorkPlan& plan,
                                   const float* ws_o, const float* ws_lse, void* out, float* lse,
                                   int32_t num_seqs, cudaStream_t st) {
  static thread_local cpattn::SplitMergeParams mp;
  std::memset(&mp, 0, sizeof(mp));
  const cpattn_config& c = ctx->cfg;
  mp.ws_o = ws_o;
  mp.ws_lse = ws_lse;
  mp.out = static_cast<__nv_bfloat16*>(out);
  mp.lse = lse;
  mp.C = c.chunk_size;
  mp.nq = c.num_q_heads;
  mp.hd = c.head_dim;
  mp.num_groups = static_cast<int>(plan.groups.size());
  long long total = 0;
  for (int g = 0; g < mp.num_groups; ++g) {
    const cpattn::SplitGroup& G = plan.groups[g];
    mp.g_b[g] = G.b;
    mp.g_q0[g] = G.q0;
    mp.g_rows[g] = G.rows;
    mp.g_n[g] = G.n;
    mp.g_part0[g] = G.part0;
    mp.g_prefix[g] = total;
    total += static_cast<long long>(G.rows) * c.num_q_heads;  // (row, head) pairs
  }
  mp.g_prefix[mp.num_groups] = total;
  mp.total = total;
  (void)num_seqs;
  // One CTA per (row, head), grid-stride beyond a few waves.
  const int grid = static_cast<int>(std::max<long long>(
      1, std::min<long long>(total, static_cast<long long>(std::max(ctx->num_sms, 1)) * 16)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(32 * cpattn::kMergeWarps, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, cpattn::splitkv_merge_kernel, mp);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "split-KV merge launch");
  return after_launch(ctx, st, "split-KV merge launch");
}

// Plan and launch one prefill: all regions (optionally split-KV, then the
// merge), or one region of the two-launch variant.  Arguments already
// validated.
cpattn_status prefill_launch(cpattn_ctx* ctx, int32_t num_seqs, const int32_t* cache_lens,
                             const int32_t* chunk_lens, const void* q, const void* k_new,
                             const void* v_new, const void* k_cache, const void* v_cache,
                             void* out, float* lse, void* stream, int region, int out_f32,
                             int split, bool write_kv = false, const void* v_cur = nullptr,
                             int cur_f16 = 0) {
  const cpattn_config& c = ctx->cfg;
  const int HD = c.head_dim, NQ = c.num_q_heads, NKV = c.num_kv_heads;
  static thread_local cpattn::WorkPlan plan;
  std::string why;
  const int block_tokens = pack_block_tokens(ctx, num_seqs, chunk_lens, region);
  const bool packed = block_tokens != kBQ;
  int executors = 0, units_per_block = 0;
  plan_shape(ctx, packed, &executors, &units_per_block);
  if (!cpattn::make_plan(c, num_seqs, cache_lens, chunk_lens, region, split, executors,
                         units_per_block, block_tokens, &plan, &why))
    return fail(ctx, CPATTN_E_UNSUPPORTED, why);
  if (plan.blocks.empty()) return CPATTN_OK;
  const size_t ws_need = cpattn::plan_workspace_bytes(plan, NQ, HD);
  if (ws_need > ctx->split_ws_bytes)
    return fail(ctx, CPATTN_E_INVALID,
                "the registered split-KV workspace holds " + std::to_string(ctx->split_ws_bytes) +
                    " bytes; this batch's plan needs " + std::to_string(ws_need) +
                    " (cpattn_splitkv_workspace)");
  if (ctx->d_status == nullptr) return fail(ctx, CPATTN_E_CUDA, "no CUDA device");

  static thread_local cpattn::PrefillParams prm;
  std::memset(&prm, 0, sizeof(prm));
  const uint64_t T = static_cast<uint64_t>(num_seqs) * c.chunk_size;
  const uint64_t rows = static_cast<uint64_t>(num_seqs) * NKV * c.num_shards * c.shard_capacity;
  const uint32_t vrows = 8192u / static_cast<uint32_t>(HD);
  const uint64_t rb = static_cast<uint64_t>(HD) * 2;
  bool ok = encode3d(&prm.tm_q, q, HD, NQ, T, rb, rb * NQ, 64, 1, kBQ) &&
            encode3d(&prm.tm_k_new, k_new, HD, NKV, T, rb, rb * NKV, 64, 1, kBKV) &&
            encode3d(&prm.tm_v_new, v_cur != nullptr ? v_cur : v_new, HD, NKV, T, rb, rb * NKV,
                     64, 1, vrows) &&
            encode3d(&prm.tm_k_cache, k_cache, HD, 1, rows, rb, rb, 64, 1, kBKV) &&
            encode3d(&prm.tm_v_cache, v_cache, HD, 1, rows, rb, rb, 64, 1, vrows) &&
            encode3d(&prm.tm_k_new_h, k_new, HD, NKV, T, rb, rb * NKV, 64, 1, kBKV / 2) &&
            encode3d(&prm.tm_k_cache_h, k_cache, HD, 1, rows, rb, rb, 64, 1, kBKV / 2) &&
            encode3d(&prm.tm_v_new_h, v_cur != nullptr ? v_cur : v_new, HD, NKV, T, rb, rb * NKV,
                     64, 1, 64) &&
            encode3d(&prm.tm_v_cache_h, v_cache, HD, 1, rows, rb, rb, 64, 1, 64) &&
            (!packed || encode3d(&prm.tm_q_packed, q, HD, NQ, T, rb, rb * NQ, 64,
                                 static_cast<uint32_t>(NQ / NKV), static_cast<uint32_t>(block_tokens)));
  if (!ok) return fail(ctx, CPATTN_E_CUDA, "cuTensorMapEncodeTiled failed");
  prm.packed = packed ? 1 : 0;
  prm.tb = block_tokens;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.lse = lse;
  prm.out_f32 = out_f32;
  if (write_kv) {
    prm.k_new = static_cast<const __nv_bfloat16*>(k_new);
    prm.v_new = static_cast<const __nv_bfloat16*>(v_new);
    prm.k_cache_w = static_cast<__nv_bfloat16*>(const_cast<void*>(k_cache));
    prm.v_cache_w = static_cast<__nv_bfloat16*>(const_cast<void*>(v_cache));
  }
  if (ws_need > 0) {
    const size_t o_bytes =
        cpattn::align256(static_cast<size_t>(plan.partial_rows) * NQ * static_cast<size_t>(HD) * 4);
    prm.ws_o = static_cast<float*>(ctx->split_ws);
    prm.ws_lse = reinterpret_cast<float*>(static_cast<char*>(ctx->split_ws) + o_bytes);
  }
  prm.status = ctx->d_status;
  prm.timeout_ns = ctx->timeout_ns;
  prm.nq = NQ;
  prm.nkv = NKV;
  prm.group = NQ / NKV;
  prm.P = c.num_shards;
  prm.S = c.shard_capacity;
  prm.C = c.chunk_size;
  prm.debug_flags = ctx->debug_flags;
  prm.scale_log2 = c.softmax_scale * 1.4426950408889634f;
  for (int b = 0; b < num_seqs; ++b)
    prm.seqs[b] = cpattn::SeqInfo{cache_lens[b], chunk_lens[b], plan.ncache[b], 0};
  // Unit order (PrefillParams::per): kv-head-major takes one block entry per
  // (row block, kv head), so it needs NKV times the entries.
  const size_t nblk = plan.blocks.size();
  bool kv_major = false;
  if (!packed && NKV > 1 && NQ <= 16384 && nblk * NKV <= CPATTN_MAX_ROW_BLOCKS &&
      ctx->unit_order != 1) {
    std::vector<int>& lens = ctx->block_lens;
    lens.clear();
    for (const cpattn::WorkBlock& b : plan.blocks) lens.push_back(b.v1 - b.v0);
    // Executors take units_per_block units of a block (q heads, or head pairs).
    kv_major = ctx->unit_order == 2 ||
               cpattn::prefer_kv_major(lens, units_per_block / NKV, NKV, executors);
  }
  const int G = NQ / NKV;
  const int reps = kv_major ? NKV : 1;
  prm.per = kv_major ? G : (packed ? NKV : NQ);
  for (int g = 0, i = 0; g < reps; ++g)
    for (size_t j = 0; j < nblk; ++j, ++i) {
      const cpattn::WorkBlock& w = plan.blocks[j];
      prm.blocks[i] = cpattn::pack_block(w.b, w.qb, g * G);
      prm.range[i] = (static_cast<uint32_t>(w.v0) << 16) | static_cast<uint32_t>(w.v1);
      prm.part[i] = w.part;
    }
  prm.num_units = static_cast<int>(nblk * reps) * prm.per;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cpattn_status s = dispatch_prefill(ctx, &prm, st, packed, cur_f16 != 0);
  if (s != CPATTN_OK || plan.groups.empty()) return s;
  return launch_splitkv_merge(ctx, plan, prm.ws_o, prm.ws_lse, out, lse, num_seqs, st);
}

// Bytes of the fp16 V staging buffer for a batch of num_seqs sequences:
// the chunk's V in token order, [num_seqs * C, NKV, HD] fp16.
uint64_t v_stage_need(const cpattn_config& c, int32_t num_seqs) {
  return static_cast<uint64_t>(num_seqs) * c.chunk_size * c.num_kv_heads * c.head_dim * 2;
}

// fp16 V cache with a registered staging buffer: launch the staging of the
// chunk's V (stage_v_f16_kernel) and point *v_cur at it, *cur_f16 = 1.
// Otherwise *v_cur = v_new (bf16) and *cur_f16 = 0.
cpattn_status stage_v(cpattn_ctx* ctx, int32_t num_seqs, const int32_t* chunk_lens,
                      const void* v_new, void* stream, const void** v_cur, int* cur_f16) {
  const cpattn_config& c = ctx->cfg;
  *v_cur = v_new;
  *cur_f16 = 0;
  if (!c.v_cache_f16 || ctx->v_stage == nullptr) return CPATTN_OK;
  const uint64_t need = v_stage_need(c, num_seqs);
  if (need > ctx->v_stage_bytes)
    return fail(ctx, CPATTN_E_INVALID,
                "the registered V staging buffer holds " + std::to_string(ctx->v_stage_bytes) +
                    " bytes; this batch needs " + std::to_string(need) +
                    " (cpattn_v_staging_bytes)");
  if (ctx->d_status == nullptr) return fail(ctx, CPATTN_E_CUDA, "no CUDA device");
  cpattn::StageVParams p;
  p.v_new = static_cast<const uint4*>(v_new);
  p.v_stage = static_cast<uint4*>(ctx->v_stage);
  p.status = ctx->d_status;
  p.C = c.chunk_size;
  p.nkv = c.num_kv_heads;
  p.vec_per_row = c.head_dim * 2 / 16;
  p.total_vecs = static_cast<long long>(need / 16);
  for (int b = 0; b < num_seqs; ++b) p.chunk_len[b] = chunk_lens[b];
  // One wave (4 blocks of 256 threads per SM, grid-stride beyond): every
  // block starts at once, so the prefill kernel, its programmatic dependent,
  // may launch as soon as the blocks have started.
  const long long blocks = (p.total_vecs + 255) / 256;
  const int grid =
      static_cast<int>(std::min<long long>(blocks, static_cast<long long>(ctx->num_sms) * 4));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cpattn::stage_v_f16_kernel<<<grid, 256, 0, st>>>(p);
  cpattn_status s = after_launch(ctx, st, "V staging launch");
  if (s != CPATTN_OK) return s;
  *v_cur = ctx->v_stage;
  *cur_f16 = 1;
  return CPATTN_OK;
}

}  // namespace

extern "C" {

const char* cpattn_status_string(cpattn_status s) {
  switch (s) {
    case CPATTN_OK: return "ok";
    case CPATTN_E_INVALID: return "invalid argument";
    case CPATTN_E_UNSUPPORTED: return "unsupported by this build";
    case CPATTN_E_CUDA: return "CUDA error";
    case CPATTN_E_NOMEM: return "out of memory";
    case CPATTN_E_TIMEOUT: return "device-side wait timed out";
    case CPATTN_E_RANGE: return "value outside the fp16 V cache's range";
  }
  return "unknown status";
}

const char* cpattn_last_error(const cpattn_ctx* ctx) {
  return ctx == nullptr ? "" : ctx->last_error.c_str();
}

// Checks of a configuration shared by cpattn_create and the allocation-free
// prefill.
static cpattn_status check_config(const cpattn_config& c) {
  if (c.num_q_heads < 1 || c.num_kv_heads < 1 || c.num_shards < 1 || c.shard_capacity < 1 ||
      c.chunk_size < 1 || c.num_q_heads % c.num_kv_heads != 0 || c.fast_p < 0 || c.fast_p > 1 ||
      c.v_cache_f16 < 0 || c.v_cache_f16 > 1 || c.pairing < 0 || c.pairing > 2 ||
      c.gqa_packing < 0 || c.gqa_packing > 1)
    return CPATTN_E_INVALID;
  if (c.head_dim != 128 && c.head_dim != 256) return CPATTN_E_UNSUPPORTED;
  // Work units are (row block, q head) and their count must fit the kernel's int.
  if (c.num_q_heads > 65535) return CPATTN_E_UNSUPPORTED;
  return CPATTN_OK;
}

cpattn_status cpattn_create(const cpattn_config* cfg, cpattn_ctx** out) {
  if (out == nullptr || cfg == nullptr) return CPATTN_E_INVALID;
  *out = nullptr;
  const cpattn_config& c = *cfg;
  const cpattn_status cs = check_config(c);
  if (cs != CPATTN_OK) return cs;
  cpattn_ctx* ctx = new (std::nothrow) cpattn_ctx();
  if (ctx == nullptr) return CPATTN_E_NOMEM;
  ctx->cfg = c;
  if (!(c.softmax_scale > 0.f)) ctx->cfg.softmax_scale = 1.0f / std::sqrt(static_cast<float>(c.head_dim));
  ctx->pair_mode = c.pairing == CPATTN_PAIRING_NONE       ? 0
                   : c.pairing == CPATTN_PAIRING_PINGPONG ? 3
                                                          : 2;
  ctx->gqa_packing = c.gqa_packing == CPATTN_GQA_PACKING_AUTO;
  const char* dbg = std::getenv("CPATTN_DEBUG");
  ctx->debug_sync = dbg != nullptr && dbg[0] == '1';
  // Test overrides of the configuration's kernel-form fields.
  const char* packing = std::getenv("CPATTN_GQA_PACKING");
  if (packing != nullptr) {
    if (std::strcmp(packing, "off") == 0) ctx->gqa_packing = false;
    else if (std::strcmp(packing, "auto") == 0) ctx->gqa_packing = true;
    else {
      delete ctx;
      return CPATTN_E_INVALID;
    }
  }
  const char* order = std::getenv("CPATTN_UNIT_ORDER");
  if (order != nullptr) {
    if (std::strcmp(order, "auto") == 0) ctx->unit_order = 0;
    else if (std::strcmp(order, "longest") == 0) ctx->unit_order = 1;
    else if (std::strcmp(order, "kv_major") == 0) ctx->unit_order = 2;
    else {
      delete ctx;
      return CPATTN_E_INVALID;
    }
  }
  const char* pairing = std::getenv("CPATTN_PAIRING");
  if (pairing != nullptr) {
    if (std::strcmp(pairing, "none") == 0) ctx->pair_mode = 0;
    else if (std::strcmp(pairing, "mma2") == 0) ctx->pair_mode = 2;
    else if (std::strcmp(pairing, "pingpong") == 0) ctx->pair_mode = 3;
    else {
      delete ctx;
      return CPATTN_E_INVALID;
    }
  }
  int dev = -1, ndev = 0;
  if (cudaGetDeviceCount(&ndev) == cudaSuccess && ndev > 0 && cudaGetDevice(&dev) == cudaSuccess) {
    ctx->device = dev;
    cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (cudaMalloc(&ctx->d_status, sizeof(int)) != cudaSuccess ||
        cudaMemset(ctx->d_status, 0, sizeof(int)) != cudaSuccess) {
      cudaFree(ctx->d_status);
      delete ctx;
      return CPATTN_E_NOMEM;
    }
  } else {
    cudaGetLastError();  // clear the "no device" error
  }
  *out = ctx;
  return CPATTN_OK;
}

void cpattn_destroy(cpattn_ctx* ctx) {
  if (ctx == nullptr) return;
  if (ctx->d_status != nullptr) cudaFree(ctx->d_status);
  delete ctx;
}

cpattn_status cpattn_set_fault_injection(cpattn_ctx* ctx, int32_t flags, int32_t timeout_ms) {
  if (ctx == nullptr || flags < 0 || flags > 1) return CPATTN_E_INVALID;
  ctx->debug_flags = flags;
  ctx->timeout_ns = timeout_ms > 0 ? static_cast<unsigned long long>(timeout_ms) * 1000000ull
                                   : 1000ull * 1000 * 1000;
  return CPATTN_OK;
}

cpattn_status cpattn_set_barrier_counts(cpattn_ctx* ctx, void* records, uint64_t bytes) {
  if (ctx == nullptr) return CPATTN_E_INVALID;
#ifdef CPATTN_COUNT_BARRIERS
  if (records != nullptr && (reinterpret_cast<uintptr_t>(records) & 3u) != 0)
    return fail(ctx, CPATTN_E_INVALID, "barrier-count records must be 4-byte aligned");
  ctx->bar_counts = static_cast<uint32_t*>(records);
  ctx->bar_counts_bytes = records != nullptr ? static_cast<size_t>(bytes) : 0;
  return CPATTN_OK;
#else
  (void)records, (void)bytes;
  return fail(ctx, CPATTN_E_UNSUPPORTED, "barrier counting needs the barrier-count build");
#endif
}

cpattn_status cpattn_cache_walk(const cpattn_ctx* ctx, int32_t cache_len, int32_t* tiles,
                                uint32_t* masks, int32_t max_tiles, int32_t* count) {
  return cpattn_cache_walk_from(ctx, cache_len, 0, tiles, masks, max_tiles, count);
}

cpattn_status cpattn_cache_walk_from(const cpattn_ctx* ctx, int32_t cache_len, int32_t first,
                                     int32_t* tiles, uint32_t* masks, int32_t max_tiles,
                                     int32_t* count) {
  if (ctx == nullptr || count == nullptr || cache_len < 0 || max_tiles < 0 || first < 0)
    return CPATTN_E_INVALID;
  const int P = ctx->cfg.num_shards, S = ctx->cfg.shard_capacity;
  if (static_cast<long long>(cache_len) > static_cast<long long>(P) * S) return CPATTN_E_INVALID;
  cpattn::CacheWalk w;
  w.init(cache_len, P, S);
  w.skip(first);  // as a split-KV piece starting at virtual tile `first` does
  int n = 0;
  while (!w.done()) {
    const int t = w.next();
    if ((tiles != nullptr || masks != nullptr) && n >= max_tiles) return CPATTN_E_INVALID;
    if (tiles != nullptr) tiles[n] = t;
    if (masks != nullptr) {
      // Same decision as the prefill kernel: interior tiles are full.
      uint32_t mw[4] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
      if (!w.last_full) w.column_mask(t, mw);
      std::memcpy(masks + 4 * n, mw, sizeof(mw));
    }
    ++n;
  }
  *count = n;
  return CPATTN_OK;
}

cpattn_status cpattn_sync_status(cpattn_ctx* ctx, void* stream) {
  if (ctx == nullptr) return CPATTN_E_INVALID;
  if (ctx->d_status == nullptr) return fail(ctx, CPATTN_E_CUDA, "no CUDA device");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaStreamSynchronize");
  int word = 0;
  e = cudaMemcpy(&word, ctx->d_status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "reading the status word");
  if (word != 0) {
    cudaMemset(ctx->d_status, 0, sizeof(int));
    if ((word & 0xFF) == cpattn::kStatusLayout)
      return fail(ctx, CPATTN_E_CUDA,
                  "the kernel's dynamic shared memory base was not aligned as required; "
                  "it returned without computing");
    if ((word & 0xFF) == cpattn::kStatusRange)
      return fail(ctx, CPATTN_E_RANGE,
                  "a V value converted to fp16 (for the fp16 V cache, or staged) lies outside "
                  "fp16's finite range");
    return fail(ctx, CPATTN_E_TIMEOUT,
                "a bounded device wait expired (site " + std::to_string(word >> 8) + ")");
  }
  return CPATTN_OK;
}

cpattn_status cpattn_write_kv(cpattn_ctx* ctx, int32_t num_seqs, const int32_t* cache_lens,
                              const int32_t* chunk_lens, const void* k_new, const void* v_new,
                              void* k_cache, void* v_cache, void* stream) {
  if (ctx == nullptr) return CPATTN_E_INVALID;
  cpattn_status s = check_seqs(ctx, num_seqs, cache_lens, chunk_lens);
  if (s != CPATTN_OK) return s;
  if (k_new == nullptr || v_new == nullptr || k_cache == nullptr || v_cache == nullptr)
    return fail(ctx, CPATTN_E_INVALID, "device pointers must not be NULL");
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(ctx, CPATTN_E_INVALID, "device pointers must be 16-byte aligned");
  const cpattn_config& c = ctx->cfg;
  cpattn::WriteKvParams p;
  p.k_new = static_cast<const uint4*>(k_new);
  p.v_new = static_cast<const uint4*>(v_new);
  p.k_cache = static_cast<uint4*>(k_cache);
  p.v_cache = static_cast<uint4*>(v_cache);
  p.status = ctx->d_status;
  p.v_f16 = c.v_cache_f16;
  p.num_seqs = num_seqs;
  p.nkv = c.num_kv_heads;
  p.P = c.num_shards;
  p.S = c.shard_capacity;
  p.C = c.chunk_size;
  p.vec_per_row = c.head_dim * 2 / 16;
  long long acc = 0;
  for (int b = 0; b < num_seqs; ++b) {
    p.cache_len[b] = cache_lens[b];
    p.vec_prefix[b] = acc;
    acc += static_cast<long long>(chunk_lens[b]) * c.num_kv_heads * p.vec_per_row;
  }
  p.vec_prefix[num_seqs] = acc;
  p.total_vecs = acc;
  if (acc == 0) return CPATTN_OK;
  if (ctx->d_status == nullptr) return fail(ctx, CPATTN_E_CUDA, "no CUDA device");
  const long long blocks = (acc + 255) / 256;
  const int grid = static_cast<int>(std::min<long long>(blocks, static_cast<long long>(ctx->num_sms) * 16));
  cpattn::write_kv_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return after_launch(ctx, static_cast<cudaStream_t>(stream), "write_kv launch");
}

cpattn_status cpattn_prefill(cpattn_ctx* ctx, int32_t num_seqs, const int32_t* cache_lens,
                             const int32_t* chunk_lens, const void* q, const void* k_new,
                             const void* v_new, const void* k_cache, const void* v_cache,
                             void* out, float* lse, void* stream) {
  if (ctx == nullptr) return CPATTN_E_INVALID;
  cpattn_status s = check_seqs(ctx, num_seqs, cache_lens, chunk_lens);
  if (s != CPATTN_OK) return s;
  if (q == nullptr || k_new == nullptr || v_new == nullptr || k_cache == nullptr ||
      v_cache == nullptr || out == nullptr)
    return fail(ctx, CPATTN_E_INVALID, "device pointers must not be NULL");
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(out) || (lse != nullptr && !aligned16(lse)))
    return fail(ctx, CPATTN_E_INVALID, "device pointers must be 16-byte aligned");
  const void* v_cur = nullptr;
  int cur_f16 = 0;
  s = stage_v(ctx, num_seqs, chunk_lens, v_new, stream, &v_cur, &cur_f16);
  if (s != CPATTN_OK) return s;
  return prefill_launch(ctx, num_seqs, cache_lens, chunk_lens, q, k_new, v_new, k_cache, v_cache,
                        out, lse, stream, cpattn::kRegionAll, 0,
                        ctx->split_ws != nullptr ? ctx->split_policy : cpattn::kSplitOff, false,
                        v_cur, cur_f16);
}

cpattn_status cpattn_prefill_write_kv(cpattn_ctx* ctx, int32_t num_seqs,
                                      const int32_t* cache_lens, const int32_t* chunk_lens,
                                      const void* q, const void* k_new, const void* v_new,
                                      void* k_cache, void* v_cache, void* out, float* lse,
                                      void* stream) {
  if (ctx == nullptr) return CPATTN_E_INVALID;
  cpattn_status s = check_seqs(ctx, num_seqs, cache_lens, chunk_lens);
  if (s != CPATTN_OK) return s;
  if (q == nullptr || k_new == nullptr || v_new == nullptr || k_cache == nullptr ||
      v_cache == nullptr || out == nullptr)
    return fail(ctx, CPATTN_E_INVALID, "device pointers must not be NULL");
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(out) || (lse != nullptr && !aligned16(lse)))
    return fail(ctx, CPATTN_E_INVALID, "device pointers must be 16-byte aligned");
  const void* v_cur = nullptr;
  int cur_f16 = 0;
  s = stage_v(ctx, num_seqs, chunk_lens, v_new, stream, &v_cur, &cur_f16);
  if (s != CPATTN_OK) return s;
  return prefill_launch(ctx, num_seqs, cache_lens, chunk_lens, q, k_new, v_new, k_cache, v_cache,
                        out, lse, stream, cpattn::kRegionAll, 0,
                        ctx->split_ws != nullptr ? ctx->split_policy : cpattn::kSplitOff, true,
                        v_cur, cur_f16);
}

cpattn_status cpattn_set_splitkv(cpattn_ctx* ctx, void* workspace, uint64_t workspace_bytes,
                                 int32_t max_split_tiles) {
  if (ctx == nullptr || max_split_tiles < 0) return CPATTN_E_INVALID;
  if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(ctx, CPATTN_E_INVALID, "split-KV workspace must be 256-byte aligned");
  ctx->split_ws = workspace;
  ctx->split_ws_bytes = workspace != nullptr ? static_cast<size_t>(workspace_bytes) : 0;
  ctx->split_policy = workspace != nullptr ? max_split_tiles : cpattn::kSplitOff;
  return CPATTN_OK;
}

cpattn_status cpattn_splitkv_workspace(const cpattn_ctx* ctx, int32_t num_seqs,
                                       const int32_t* cache_lens, const int32_t* chunk_lens,
                                       int32_t max_split_tiles, uint64_t* bytes,
                                       int32_t* work_blocks) {
  if (ctx == nullptr || bytes == nullptr || max_split_tiles < 0) return CPATTN_E_INVALID;
  cpattn_status s = check_seqs(const_cast<cpattn_ctx*>(ctx), num_seqs, cache_lens, chunk_lens);
  if (s != CPATTN_OK) return s;
  cpattn::WorkPlan plan;
  std::string why;
  const int block_tokens = pack_block_tokens(ctx, num_seqs, chunk_lens, cpattn::kRegionAll);
  int executors = 0, units_per_block = 0;
  plan_shape(ctx, block_tokens != kBQ, &executors, &units_per_block);
  if (!cpattn::make_plan(ctx->cfg, num_seqs, cache_lens, chunk_lens, cpattn::kRegionAll,
                         max_split_tiles, executors, units_per_block, block_tokens, &plan, &why))
    return CPATTN_E_UNSUPPORTED;
  *bytes = cpattn::plan_workspace_bytes(plan, ctx->cfg.num_q_heads, ctx->cfg.head_dim);
  if (work_blocks != nullptr) *work_blocks = static_cast<int32_t>(plan.blocks.size());
  return CPATTN_OK;
}

cpattn_status cpattn_set_v_staging(cpattn_ctx* ctx, void* buffer, uint64_t bytes) {
  if (ctx == nullptr) return CPATTN_E_INVALID;
  if (buffer != nullptr && !ctx->cfg.v_cache_f16)
    return fail(ctx, CPATTN_E_INVALID, "V staging applies to an fp16 V cache only");
  if (buffer != nullptr && !aligned16(buffer))
    return fail(ctx, CPATTN_E_INVALID, "the V staging buffer must be 16-byte aligned");
  ctx->v_stage = buffer;
  ctx->v_stage_bytes = buffer != nullptr ? static_cast<size_t>(bytes) : 0;
  return CPATTN_OK;
}

cpattn_status cpattn_v_staging_bytes(const cpattn_ctx* ctx, int32_t num_seqs, uint64_t* bytes) {
  if (ctx == nullptr || bytes == nullptr || num_seqs < 1 || num_seqs > CPATTN_MAX_SEQS)
    return CPATTN_E_INVALID;
  *bytes = v_stage_need(ctx->cfg, num_seqs);
  return CPATTN_OK;
}

// Two-launch variant: workspace = two fp32 partial outputs and two LSE rows.
static uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

static void two_launch_layout(const cpattn_config& c, int32_t num_seqs, uint64_t off[4],
                              uint64_t* total) {
  const uint64_t T = static_cast<uint64_t>(num_seqs) * c.chunk_size;
  const uint64_t o = align256(T * c.num_q_heads * c.head_dim * sizeof(float));
  const uint64_t l = align256(T * c.num_q_heads * sizeof(float));
  off[0] = 0;
  off[1] = o;
  off[2] = 2 * o;
  off[3] = 2 * o + l;
  *total = 2 * o + 2 * l;
}

cpattn_status cpattn_two_launch_workspace(const cpattn_ctx* ctx, int32_t num_seqs,
                                          uint64_t* bytes) {
  if (ctx == nullptr || bytes == nullptr || num_seqs < 1) return CPATTN_E_INVALID;
  uint64_t off[4];
  two_launch_layout(ctx->cfg, num_seqs, off, bytes);
  return CPATTN_OK;
}

cpattn_status cpattn_prefill_two_launch(cpattn_ctx* ctx, int32_t num_seqs,
                                        const int32_t* cache_lens, const int32_t* chunk_lens,
                                        const void* q, const void* k_new, const void* v_new,
                                        const void* k_cache, const void* v_cache, void* out,
                                        float* lse, void* workspace, uint64_t workspace_bytes,
                                        void* stream) {
  if (ctx == nullptr) return CPATTN_E_INVALID;
  cpattn_status s = check_seqs(ctx, num_seqs, cache_lens, chunk_lens);
  if (s != CPATTN_OK) return s;
  if (q == nullptr || k_new == nullptr || v_new == nullptr || k_cache == nullptr ||
      v_cache == nullptr || out == nullptr || workspace == nullptr)
    return fail(ctx, CPATTN_E_INVALID, "device pointers must not be NULL");
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(out) || (lse != nullptr && !aligned16(lse)) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(ctx, CPATTN_E_INVALID, "pointer alignment (16 B; workspace 256 B)");
  const cpattn_config& c = ctx->cfg;
  uint64_t off[4], need;
  two_launch_layout(c, num_seqs, off, &need);
  if (workspace_bytes < need)
    return fail(ctx, CPATTN_E_INVALID,
                "workspace too small: need " + std::to_string(need) + " bytes");
  char* ws = static_cast<char*>(workspace);
  float* o1 = reinterpret_cast<float*>(ws + off[0]);
  float* o2 = reinterpret_cast<float*>(ws + off[1]);
  float* l1 = reinterpret_cast<float*>(ws + off[2]);
  float* l2 = reinterpret_cast<float*>(ws + off[3]);
  // Launch 1: cache tiles only; launch 2: current tiles only (causal).  The
  // tiles take the fused launch's forms (with a staged fp16 V, every tile
  // fp16 P and one P.V product).
  const void* v_cur = nullptr;
  int cur_f16 = 0;
  s = stage_v(ctx, num_seqs, chunk_lens, v_new, stream, &v_cur, &cur_f16);
  if (s != CPATTN_OK) return s;
  s = prefill_launch(ctx, num_seqs, cache_lens, chunk_lens, q, k_new, v_new, k_cache, v_cache,
                     o1, l1, stream, cpattn::kRegionCache, 1, cpattn::kSplitOff, false, v_cur,
                     cur_f16);
  if (s != CPATTN_OK) return s;
  s = prefill_launch(ctx, num_seqs, cache_lens, chunk_lens, q, k_new, v_new, k_cache, v_cache,
                     o2, l2, stream, cpattn::kRegionCurrent, 1, cpattn::kSplitOff, false, v_cur,
                     cur_f16);
  if (s != CPATTN_OK) return s;
  // Launch 3: LSE merge into bf16 O.
  cpattn::MergeParams m;
  m.o1 = o1;
  m.lse1 = l1;
  m.o2 = o2;
  m.lse2 = l2;
  m.out = static_cast<__nv_bfloat16*>(out);
  m.lse = lse;
  m.num_seqs = num_seqs;
  m.C = c.chunk_size;
  m.nq = c.num_q_heads;
  m.hd = c.head_dim;
  long long acc = 0;
  for (int b = 0; b < num_seqs; ++b) {
    m.has_cache[b] = cache_lens[b] > 0 ? 1 : 0;
    m.item_prefix[b] = acc;
    acc += static_cast<long long>(chunk_lens[b]) * c.num_q_heads * (c.head_dim / 8);
  }
  m.item_prefix[num_seqs] = acc;
  m.total = acc;
  if (acc == 0) return CPATTN_OK;
  const long long blocks = (acc + 255) / 256;
  const int grid = static_cast<int>(std::min<long long>(blocks, static_cast<long long>(ctx->num_sms) * 16));
  cpattn::lse_merge_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(m);
  return after_launch(ctx, static_cast<cudaStream_t>(stream), "merge launch");
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free prefill.  Some callers must not allocate device memory at
// all: code that runs while a custom or pooled allocator owns the device,
// code inside a region where cudaMalloc/cudaFree would synchronise the device
// or are forbidden (for instance while a stream is being captured), and
// embedders that only hand over input and output pointers.  The context-based
// cpattn_prefill needs cpattn_create, which cudaMalloc's the kernel's status
// word; this entry point instead keeps that scratch word in the file-scope
// array below, which every GPU that loads the library holds until exit.

// Scratch of the allocation-free path: word 0 is the prefill kernel's
// bounded-wait status word.  256 bytes per device.
static __device__ __align__(256) int g_noalloc_scratch[CPATTN_NOALLOC_SCRATCH_INTS];

namespace {

constexpr int kNoAllocMaxDevices = 64;

// The unpaired kernel of one precision form, as the allocation-free entry
// point launches it (plain launch, no cluster).
template <int HD, bool SPLIT, bool VF16>
cudaError_t noalloc_attr() {
  const void* k = reinterpret_cast<const void*>(cpattn::prefill_kernel<HD, SPLIT, VF16>);
  if (cpattn::Layout<HD>::SPLIT_O && !register_split_ok(k)) return cudaErrorInvalidDeviceFunction;
  return cudaFuncSetAttribute(cpattn::prefill_kernel<HD, SPLIT, VF16>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              cpattn::Layout<HD>::SMEM_BYTES);
}
template <int HD, bool SPLIT, bool VF16>
void noalloc_launch(int grid, cudaStream_t st, const cpattn::PrefillParams& prm) {
  cpattn::prefill_kernel<HD, SPLIT, VF16>
      <<<grid, cpattn::kThreads, cpattn::Layout<HD>::SMEM_BYTES, st>>>(prm);
}

struct NoAllocDevice {
  bool ready = false;
  int* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int num_sms = 0;
};

NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];
std::mutex g_noalloc_mutex;

// Once per device, with that device current: resolve the device address of
// the scratch array (its host-side name is only a stand-in) and set the
// kernels' shared-memory attribute.
cpattn_status noalloc_setup(NoAllocDevice** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return CPATTN_E_CUDA;
  if (dev >= kNoAllocMaxDevices) return CPATTN_E_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoAllocDevice& d = g_noalloc_dev[dev];
  if (!d.ready) {
    int* ptr = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_scratch) != cudaSuccess ||
        ptr == nullptr)
      return CPATTN_E_CUDA;
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return CPATTN_E_CUDA;
    if (noalloc_attr<128, true, false>() != cudaSuccess ||
        noalloc_attr<128, false, false>() != cudaSuccess ||
        noalloc_attr<256, true, false>() != cudaSuccess ||
        noalloc_attr<256, false, false>() != cudaSuccess ||
        noalloc_attr<128, true, true>() != cudaSuccess ||
        noalloc_attr<128, false, true>() != cudaSuccess ||
        noalloc_attr<256, true, true>() != cudaSuccess ||
        noalloc_attr<256, false, true>() != cudaSuccess)
      return CPATTN_E_CUDA;
    d.scratch = ptr;
    d.ready = true;
  }
  *out = &d;
  return CPATTN_OK;
}

// True iff p is device (or managed) memory known to the driver; a host or
// truncated address is refused before it can reach a kernel.
bool is_device_ptr(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

}  // namespace

extern "C" cpattn_status cpattn_prefill_noalloc(const cpattn_config* cfg, int32_t num_seqs,
                                                const int32_t* cache_lens,
                                                const int32_t* chunk_lens, const void* q,
                                                const void* k_new, const void* v_new,
                                                const void* k_cache, const void* v_cache,
                                                void* out, float* lse, void* stream) {
  if (cfg == nullptr) return CPATTN_E_INVALID;
  const cpattn_config& c = *cfg;
  const cpattn_status cs = check_config(c);
  if (cs != CPATTN_OK) return cs;
  // Fixed-capacity host tables: sizes beyond them are refused, not grown.
  if (num_seqs < 1) return CPATTN_E_INVALID;
  if (num_seqs > CPATTN_MAX_SEQS) return CPATTN_E_UNSUPPORTED;
  if (cache_lens == nullptr || chunk_lens == nullptr || q == nullptr || k_new == nullptr ||
      v_new == nullptr || k_cache == nullptr || v_cache == nullptr || out == nullptr)
    return CPATTN_E_INVALID;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(out) || (lse != nullptr && !aligned16(lse)))
    return CPATTN_E_INVALID;
  const long long cap = static_cast<long long>(c.num_shards) * c.shard_capacity;
  int nblk = 0;
  for (int b = 0; b < num_seqs; ++b) {
    if (cache_lens[b] < 0 || chunk_lens[b] < 0 || chunk_lens[b] > c.chunk_size ||
        static_cast<long long>(cache_lens[b]) + chunk_lens[b] > cap)
      return CPATTN_E_INVALID;
    nblk += (chunk_lens[b] + kBQ - 1) / kBQ;
  }
  if (nblk > CPATTN_MAX_ROW_BLOCKS) return CPATTN_E_UNSUPPORTED;
  const long long cache_rows =
      static_cast<long long>(num_seqs) * c.num_kv_heads * c.num_shards * c.shard_capacity;
  if (cache_rows + kBKV >= (1LL << 31) ||
      static_cast<long long>(num_seqs) * c.chunk_size + kBQ >= (1LL << 31))
    return CPATTN_E_UNSUPPORTED;
  if (nblk == 0) return CPATTN_OK;

  NoAllocDevice* dev = nullptr;
  cpattn_status s = noalloc_setup(&dev);
  if (s != CPATTN_OK) return s;
  if (!is_device_ptr(q) || !is_device_ptr(k_new) || !is_device_ptr(v_new) ||
      !is_device_ptr(k_cache) || !is_device_ptr(v_cache) || !is_device_ptr(out) ||
      (lse != nullptr && !is_device_ptr(lse)))
    return CPATTN_E_INVALID;

  static thread_local cpattn::PrefillParams prm;
  static thread_local uint64_t keys[CPATTN_MAX_ROW_BLOCKS];
  std::memset(&prm, 0, sizeof(prm));
  // Row blocks longest first (ties by sequence, then block), without a heap.
  int n = 0;
  for (int b = 0; b < num_seqs; ++b) {
    const int ncache = cpattn::cache_tile_count(cache_lens[b], c.num_shards, c.shard_capacity);
    prm.seqs[b] = cpattn::SeqInfo{cache_lens[b], chunk_lens[b], ncache, 0};
    const int nqb = (chunk_lens[b] + kBQ - 1) / kBQ;
    for (int qb = 0; qb < nqb; ++qb) {
      const uint64_t work = static_cast<uint64_t>(ncache + qb + 1);
      keys[n++] = ((0xFFFFFFFFull - work) << 32) | (static_cast<uint64_t>(b) << 16) |
                  static_cast<uint64_t>(qb);
    }
  }
  std::sort(keys, keys + n);
  for (int i = 0; i < n; ++i) {
    const uint64_t work = 0xFFFFFFFFull - (keys[i] >> 32);  // whole walk: [0, n_cache + qb + 1)
    if (work > static_cast<uint64_t>(cpattn::kMaxVirtualTiles)) return CPATTN_E_UNSUPPORTED;
    prm.blocks[i] = cpattn::pack_block(static_cast<int>((keys[i] >> 16) & 0xFFFFu),
                                       static_cast<int>(keys[i] & 0xFFFFu), 0);
    prm.range[i] = static_cast<uint32_t>(work);
    prm.part[i] = -1;
  }

  const int HD = c.head_dim, NQ = c.num_q_heads, NKV = c.num_kv_heads;
  const uint64_t T = static_cast<uint64_t>(num_seqs) * c.chunk_size;
  const uint64_t rows = static_cast<uint64_t>(cache_rows);
  const uint32_t vrows = 8192u / static_cast<uint32_t>(HD);
  const uint64_t rb = static_cast<uint64_t>(HD) * 2;
  if (!(encode3d(&prm.tm_q, q, HD, NQ, T, rb, rb * NQ, 64, 1, kBQ) &&
        encode3d(&prm.tm_k_new, k_new, HD, NKV, T, rb, rb * NKV, 64, 1, kBKV) &&
        encode3d(&prm.tm_v_new, v_new, HD, NKV, T, rb, rb * NKV, 64, 1, vrows) &&
        encode3d(&prm.tm_k_cache, k_cache, HD, 1, rows, rb, rb, 64, 1, kBKV) &&
        encode3d(&prm.tm_v_cache, v_cache, HD, 1, rows, rb, rb, 64, 1, vrows)))
    return CPATTN_E_CUDA;
  const float scale = c.softmax_scale > 0.f ? c.softmax_scale
                                            : 1.0f / std::sqrt(static_cast<float>(HD));
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.lse = lse;
  prm.status = dev->scratch;
  prm.timeout_ns = 1000ull * 1000 * 1000;
  prm.nq = NQ;
  prm.nkv = NKV;
  prm.group = NQ / NKV;
  prm.P = c.num_shards;
  prm.S = c.shard_capacity;
  prm.C = c.chunk_size;
  prm.debug_flags = 0;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.per = NQ;
  prm.num_units = n * NQ;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The status word must start at zero; the previous call's value is stale.
  if (cudaMemsetAsync(dev->scratch, 0, sizeof(int), st) != cudaSuccess) return CPATTN_E_CUDA;
  const int grid = std::min(prm.num_units, dev->num_sms);
  const bool split = c.fast_p == 0;
  const bool vf16 = c.v_cache_f16 != 0;
  if (HD == 256) {
    if (vf16) split ? noalloc_launch<256, true, true>(grid, st, prm) : noalloc_launch<256, false, true>(grid, st, prm);
    else split ? noalloc_launch<256, true, false>(grid, st, prm) : noalloc_launch<256, false, false>(grid, st, prm);
  } else {
    if (vf16) split ? noalloc_launch<128, true, true>(grid, st, prm) : noalloc_launch<128, false, true>(grid, st, prm);
    else split ? noalloc_launch<128, true, false>(grid, st, prm) : noalloc_launch<128, false, false>(grid, st, prm);
  }
  return cudaGetLastError() == cudaSuccess ? CPATTN_OK : CPATTN_E_CUDA;
}
