/*
 * cpattn -- chunked-prefill GQA attention for GB300 (sm_103a), C ABI.
 *
 * One prefill step of a long-context request: a new chunk of queries attends
 * to (a) its sequence's already-cached KV prefix, fully visible, and (b) its
 * own chunk's KV under a causal mask -- both walked by ONE kernel with ONE
 * shared online softmax, with no second launch and no log-sum-exp merge
 * (TPU PR "PCP: in-kernel ring cache phase, fused with the current phase",
 * Summary and Design sections).  The PR's ring of cache shards over chips
 * becomes, on one GPU, only the iteration order over a striped cache layout.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - bf16 tensors are raw device pointers to row-major, densely packed data;
 *    every device base pointer must be 16-byte aligned.
 *  - "token order" arrays hold B*C rows: sequence b's chunk occupies rows
 *    [b*C, b*C + C); its first c_b rows are valid, the rest are padding.
 *  - Striped cache layout [B, NKV, P, S, HD]: token t of sequence b, kv head
 *    g lives in shard t mod P at row t div P (stripe width one token; the
 *    PR's "striped" shards and "strided" cache write, Design and Testing
 *    sections).  Shard s holds n_s(L) = #{t < L : t mod P = s} filled rows.
 *  - GQA: query head h reads kv head h / (NQ/NKV).
 *  - Memory the kernels may touch but must ignore (cache rows beyond the
 *    filled ones, padding rows) must hold FINITE values; non-finite values
 *    there are undefined behaviour.
 *  - Host arrays (cache_lens, chunk_lens) are read during the call only.
 *  - The caller owns every buffer.  Calls are asynchronous on `stream` (a
 *    cudaStream_t passed as void*); the library never synchronises except in
 *    cpattn_sync_status, or after each launch when the environment variable
 *    CPATTN_DEBUG=1 is set.
 *  - All argument checks run on the host before any launch; a failed check
 *    launches nothing.  No C++ exception crosses this interface.
 */
#ifndef CPATTN_H_
#define CPATTN_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CPATTN_OK = 0,
  CPATTN_E_INVALID = 1,      /* bad argument: NULL, misaligned, out-of-range size */
  CPATTN_E_UNSUPPORTED = 2,  /* valid but outside what this build handles */
  CPATTN_E_CUDA = 3,         /* a CUDA runtime/driver call or launch failed */
  CPATTN_E_NOMEM = 4,        /* host or device allocation failed (create only) */
  CPATTN_E_TIMEOUT = 5,      /* a device-side bounded wait expired; context still usable */
  CPATTN_E_RANGE = 6         /* a V value converted to fp16 (fp16 V cache or V staging)
                                lies outside fp16's range */
} cpattn_status;

typedef struct {
  int32_t num_q_heads;     /* NQ >= 1 */
  int32_t num_kv_heads;    /* NKV >= 1, NQ % NKV == 0 */
  int32_t head_dim;        /* HD: 128 or 256 */
  int32_t num_shards;      /* P >= 1 */
  int32_t shard_capacity;  /* S >= 1 rows per shard per (sequence, kv head) */
  int32_t chunk_size;      /* C >= 1 padded rows per sequence */
  float softmax_scale;     /* <= 0 selects 1/sqrt(HD) */
  int32_t fast_p;          /* 0 (default): the probabilities P enter P.V as a
                              bf16 hi + lo pair (two tensor-core products, ~16
                              significant bits); 1: P rounded once to bf16 (one
                              product, 1.5x fewer MMA FLOPs, relative RMS error
                              about 2.2e-3 instead of 1.7e-3 on N(0,1) inputs) */
  int32_t v_cache_f16;     /* 0 (default): the V cache holds bf16, as k_cache;
                              1: the V cache holds fp16.  cpattn_write_kv then
                              converts each bf16 value of v_new to fp16 (round
                              to nearest even): exact for 2^-17 <= |v| <= 65504;
                              smaller values round to a multiple of 2^-24
                              (fp16's subnormal step; |v| <= 2^-25 becomes 0),
                              an absolute error of at most 2^-25 that is not
                              reported; a value beyond 65504 is reported by the
                              next cpattn_sync_status as CPATTN_E_RANGE.
                              Prefill then takes P in fp16 for cache tiles: one
                              P.V product (11-bit P, relative RMS error about
                              1.7e-3 on N(0,1) inputs, as the bf16 hi + lo
                              pair) at the cost of fast_p.  Current-chunk tiles
                              read bf16 v_new and follow fast_p -- unless a V
                              staging buffer is registered
                              (cpattn_set_v_staging): the chunk's V is then
                              staged in fp16 and its tiles take fp16 P too. */
  int32_t pairing;         /* how prefill pairs adjacent q heads of one kv
                              head when NQ/NKV is even (results meet the same
                              accuracy in every form; the bits may differ):
                              CPATTN_PAIRING_MMA2 (0, default): a CTA pair on
                                the two SMs of a TPC runs 2-SM tensor-core MMAs
                                (M = 256) and each SM stages half of every K/V
                                tile;
                              CPATTN_PAIRING_NONE: one CTA per (q head, row
                                block);
                              CPATTN_PAIRING_PINGPONG: HD = 128 only (MMA2 at
                                HD = 256): one CTA holds both heads' query tiles
                                and alternates their products with their
                                softmaxes. */
  int32_t gqa_packing;     /* CPATTN_GQA_PACKING_AUTO (0, default): launches
                              whose chunks are all short run GQA-packed (see
                              cpattn_prefill); CPATTN_GQA_PACKING_OFF: never */
} cpattn_config;

#define CPATTN_PAIRING_MMA2 0
#define CPATTN_PAIRING_NONE 1
#define CPATTN_PAIRING_PINGPONG 2
#define CPATTN_GQA_PACKING_AUTO 0
#define CPATTN_GQA_PACKING_OFF 1

typedef struct cpattn_ctx cpattn_ctx; /* opaque */

/* Limits of this build (checked on the host). */
#define CPATTN_MAX_SEQS 128
#define CPATTN_MAX_ROW_BLOCKS 2048  /* sum over sequences of ceil(c_b / 128) */

/*
 * Create a context for one attention layer shape.
 * cfg: host pointer, read during the call.  *out receives the context.
 * Allocates a few bytes of device memory for the timeout status word on the
 * current device (skipped, without error, when no device is present; launches
 * then fail with CPATTN_E_CUDA).
 * The kernel form comes from cfg->pairing and cfg->gqa_packing.  For tests,
 * the environment variables CPATTN_PAIRING ("mma2", "none", "pingpong") and
 * CPATTN_GQA_PACKING ("auto", "off"), when set, override those two fields,
 * and CPATTN_UNIT_ORDER ("auto", "longest", "kv_major") overrides the order
 * in which prefill deals its work units (see cpattn_prefill); they are read
 * here.
 * Errors: E_INVALID (NULL, NQ % NKV != 0, sizes < 1, a field out of range,
 * an unknown CPATTN_PAIRING or CPATTN_GQA_PACKING value), E_UNSUPPORTED (HD
 * not 128/256, NQ > 65535), E_NOMEM.
 */
cpattn_status cpattn_create(const cpattn_config* cfg, cpattn_ctx** out);

/*
 * Strided KV-cache write (the PR's Testing section: the write that must be
 * bit-exact).  For every sequence b, valid chunk row i < c_b (token position
 * t = L_b + i) and kv head g:
 *   k_cache[b, g, t mod P, t div P, :] = k_new[b*C + i, g, :]   (same for V)
 * A pure bit copy, except that an fp16 V cache (cpattn_config.v_cache_f16)
 * receives each V value converted to fp16 (round to nearest even); a value
 * beyond fp16's finite range makes the next cpattn_sync_status return
 * CPATTN_E_RANGE.  Pad rows are not written; no other cache row is touched.
 *   num_seqs            B, 1..CPATTN_MAX_SEQS
 *   cache_lens[B]       host int32, L_b >= 0
 *   chunk_lens[B]       host int32, 0 <= c_b <= C, and L_b + c_b <= P*S
 *   k_new, v_new        device bf16 [B*C, NKV, HD], token order
 *   k_cache             device bf16 [B, NKV, P, S, HD], written in place
 *   v_cache             the same, bf16 or (v_cache_f16) fp16
 * Errors: E_INVALID, E_CUDA.
 */
cpattn_status cpattn_write_kv(cpattn_ctx* ctx, int32_t num_seqs, const int32_t* cache_lens,
                              const int32_t* chunk_lens, const void* k_new, const void* v_new,
                              void* k_cache, void* v_cache, void* stream);

/*
 * Fused chunked prefill (the PR's Summary and Design sections): for every
 * sequence b, query head h, valid row i < c_b,
 *   O[b*C+i, h, :] = softmax_k( scale * <q_i, k_k> ) . v_k
 * over keys k = {cache tokens 0..L_b-1} U {chunk tokens 0..i} of kv head
 * h/(NQ/NKV), as one softmax (bf16 inputs, fp32 accumulation, bf16 output).
 * Cache tokens are read from rows [0, n_s(L_b)) of each shard; the chunk's
 * own K/V come from k_new/v_new in token order.  write_kv for the same chunk
 * may run before or after this call.
 *   q                   device bf16 [B*C, NQ, HD], token order
 *   k_new, v_new        device bf16 [B*C, NKV, HD]
 *   k_cache             device bf16 [B, NKV, P, S, HD]
 *   v_cache             the same, bf16 or (v_cache_f16) fp16
 *   out                 device bf16 [B*C, NQ, HD]; pad rows are not written
 *   lse                 device fp32 [B*C, NQ] natural-log sum-exp of the
 *                       scaled logits, or NULL; pad rows not written
 * Launches whose chunks are all short (every c_b <= 64) with a power-of-two
 * group size G = NQ/NKV in [2, 128] run GQA-packed: a work unit's 128
 * query rows are 128/G tokens x the G q heads of one kv head, instead of
 * 128 tokens of one q head, so a decode step fills the tensor-core tile
 * instead of one row of it.
 * Precision of P in P.V: with a bf16 V cache, P is carried as a bf16 hi + lo
 * pair (fast_p: P rounded once to bf16); with an fp16 V cache, cache tiles
 * take P in fp16 against the fp16 V, and current-chunk tiles follow fast_p
 * -- or, with a V staging buffer registered (cpattn_set_v_staging), take P
 * in fp16 against the chunk's V staged in fp16: a kernel that converts the
 * valid rows of v_new (as cpattn_write_kv converts them; a value beyond
 * 65504 is reported by cpattn_sync_status as CPATTN_E_RANGE) runs first on
 * the stream.
 * Work units (one q head, or a pair, of one row block) go to a persistent
 * grid longest first; when the batch has several rounds of units and more
 * than one kv head, they may instead go kv-head-major (every unit of kv head
 * 0, then of kv head 1, ...) so that the units running together share one
 * kv head's K/V in L2 -- chosen when a model of the grid says it costs at
 * most 1 % of the time.  Results meet the same accuracy in either order.
 * One kernel launch -- preceded by the V staging kernel when a V staging
 * buffer is registered, and followed by a merge kernel on the same stream
 * when a split-KV workspace is registered (cpattn_set_splitkv) and the
 * batch's plan cuts some walks.
 * Errors: E_INVALID (also: the registered split-KV workspace or V staging
 * buffer is smaller than the batch needs), E_UNSUPPORTED (more than CPATTN_MAX_ROW_BLOCKS row blocks,
 * a walk of more than 65535 tiles), E_CUDA.  A device-side timeout is
 * reported by cpattn_sync_status.
 */
cpattn_status cpattn_prefill(cpattn_ctx* ctx, int32_t num_seqs, const int32_t* cache_lens,
                             const int32_t* chunk_lens, const void* q, const void* k_new,
                             const void* v_new, const void* k_cache, const void* v_cache,
                             void* out, float* lse, void* stream);

/*
 * cpattn_prefill and cpattn_write_kv of the same chunk in ONE launch (the
 * KV write fused into the prefill kernel).  A dedicated writer warp of each
 * CTA copies the chunk's valid K/V rows into the striped caches while the
 * prefill runs.  The copy writes what cpattn_write_kv writes (bits, and V
 * converted for an fp16 V cache): every (token, kv head) once, pad rows and
 * every other cache row untouched.  It
 * cannot race the prefill: it writes only rows of tokens >= L_b, which the
 * prefill never reads as keys.  Cache tiles at a shard's edge may load those
 * rows as masked columns, and they hold finite values before and after.
 * Arguments, layouts and errors are those of cpattn_prefill, with k_cache
 * and v_cache also written (in place); a registered split-KV workspace and
 * a registered V staging buffer are used as by cpattn_prefill (the staging
 * kernel runs first; the writer warp still reads the bf16 v_new).
 */
cpattn_status cpattn_prefill_write_kv(cpattn_ctx* ctx, int32_t num_seqs,
                                      const int32_t* cache_lens, const int32_t* chunk_lens,
                                      const void* q, const void* k_new, const void* v_new,
                                      void* k_cache, void* v_cache, void* out, float* lse,
                                      void* stream);

/*
 * The two-launch variant the PR removed (Summary section: a cache-only launch
 * plus an LSE merge, strictly slower than the fused kernel), kept to measure
 * what fusion saves: launch 1 attends every valid row to the cache only,
 * launch 2 to its own chunk only (causal), each writing fp32 partial O and
 * LSE into `workspace`; launch 3 merges them into bf16 `out` (and `lse`):
 *   O = (e^{l1-m} O1 + e^{l2-m} O2) / (e^{l1-m} + e^{l2-m}),  m = max(l1, l2).
 * Same arguments and result as cpattn_prefill, plus a caller-owned device
 * workspace of at least cpattn_two_launch_workspace() bytes, 256-byte
 * aligned, used only during the call's kernels on `stream`.  With a
 * registered V staging buffer the chunk's V is staged once, before launch 1,
 * and both launches take the fused launch's tile forms.
 * Errors: as cpattn_prefill; E_INVALID also for a small or misaligned workspace.
 */
cpattn_status cpattn_two_launch_workspace(const cpattn_ctx* ctx, int32_t num_seqs,
                                          uint64_t* bytes);
cpattn_status cpattn_prefill_two_launch(cpattn_ctx* ctx, int32_t num_seqs,
                                        const int32_t* cache_lens, const int32_t* chunk_lens,
                                        const void* q, const void* k_new, const void* v_new,
                                        const void* k_cache, const void* v_cache, void* out,
                                        float* lse, void* workspace, uint64_t workspace_bytes,
                                        void* stream);

/*
 * Split-KV for small chunks and decode.  With few row blocks (a short chunk,
 * or a decode step of one token) most SMs would idle while a few units walk
 * a long cache.  Once a workspace is registered here, cpattn_prefill may cut
 * a row block's tile walk (its cache tiles, then its causal current tiles)
 * into pieces run on different SMs.  Each piece writes fp32 O / l and its LSE
 * for the block's valid rows into the workspace.  A second kernel on the same
 * stream combines the pieces of each row by their LSE (the merge of the
 * two-launch variant above, generalised to n pieces) into bf16 `out` and `lse`.
 * The result is the same softmax over the same keys.  This is the single-GPU
 * counterpart of the pages' spilled running (m, l, acc) for very long
 * contexts (PCP ring-cache PR, Design section).
 *   workspace        device memory owned by the caller, 256-byte aligned,
 *                    used by every later cpattn_prefill of this context on
 *                    its stream until replaced; NULL turns split-KV off
 *                    (the default).  Calls that overlap on the GPU must not
 *                    share one workspace.
 *   workspace_bytes  its size; a prefill whose plan needs more fails with
 *                    E_INVALID (query the need with cpattn_splitkv_workspace)
 *   max_split_tiles  0: automatic -- a cost model of the persistent grid
 *                    (units handed out cyclically, longest first, each
 *                    costing its tiles plus a fixed fill/drain) picks, among
 *                    pieces of ceil(n_max / k) tiles (k = 2..64, at least 8
 *                    tiles), the cut with the lowest modelled makespan, and
 *                    cuts only if that beats the unsplit plan by 10 %;
 *                    > 0: every walk longer than this many tiles is cut into
 *                    pieces of at most this many (for tests and tuning)
 * Limits: at most 256 row blocks are cut per call (the longest ones), and
 * the pieces count against CPATTN_MAX_ROW_BLOCKS.
 * Errors: E_INVALID (NULL ctx, max_split_tiles < 0, misaligned workspace).
 */
cpattn_status cpattn_set_splitkv(cpattn_ctx* ctx, void* workspace, uint64_t workspace_bytes,
                                 int32_t max_split_tiles);

/*
 * fp16 V cache: register a device buffer owned by the caller in which
 * cpattn_prefill, cpattn_prefill_write_kv and cpattn_prefill_two_launch stage
 * the chunk's V in fp16 before their prefill kernels, so that every tile,
 * not only the cache's, takes P in fp16 with one P.V product (the cache's
 * tiles already read fp16 V).  The staging is a second kernel on the same
 * stream: valid rows of v_new converted to fp16 (round to nearest even,
 * exact for 2^-17 <= |v| <= 65504, as cpattn_write_kv converts them; a
 * value beyond 65504 is reported by cpattn_sync_status as CPATTN_E_RANGE),
 * pad rows written as zeros.
 *   buffer   device memory, 16-byte aligned, [num_seqs * C, NKV, HD] fp16
 *            for the largest batch, used by every later prefill of this
 *            context until replaced; NULL (the default) turns staging off.
 *            Calls that overlap on the GPU must not share one buffer.
 *   bytes    its size; a prefill whose batch needs more fails with
 *            E_INVALID (query the need with cpattn_v_staging_bytes)
 * cpattn_prefill_noalloc never stages (its current tiles keep the bf16 hi +
 * lo pair, or fast_p).
 * Errors: E_INVALID (NULL ctx; a buffer for a context whose V cache is
 * bf16; a misaligned buffer).
 */
cpattn_status cpattn_set_v_staging(cpattn_ctx* ctx, void* buffer, uint64_t bytes);

/*
 * Bytes of the V staging buffer for a batch of num_seqs sequences:
 * num_seqs * C * NKV * HD * 2, written to *bytes.  Host only.
 * Errors: E_INVALID (NULL ctx or bytes, num_seqs outside
 * [1, CPATTN_MAX_SEQS]).
 */
cpattn_status cpattn_v_staging_bytes(const cpattn_ctx* ctx, int32_t num_seqs, uint64_t* bytes);

/*
 * Workspace bytes the split-KV plan of this batch needs under the policy
 * `max_split_tiles` (as in cpattn_set_splitkv), written to *bytes (0 when
 * nothing would be split).  *work_blocks (if not NULL) receives the number of
 * work blocks the kernel would run: the row blocks, plus one for every extra
 * piece.  Host only; reads the sequence arrays during the call.
 * Errors: E_INVALID (as cpattn_prefill's sequence checks, NULL bytes),
 * E_UNSUPPORTED (the plan exceeds the kernel's tables).
 */
cpattn_status cpattn_splitkv_workspace(const cpattn_ctx* ctx, int32_t num_seqs,
                                       const int32_t* cache_lens, const int32_t* chunk_lens,
                                       int32_t max_split_tiles, uint64_t* bytes,
                                       int32_t* work_blocks);

/*
 * Synchronise `stream`, then read and clear the context's device status word.
 * Returns E_TIMEOUT if a kernel launched with this context gave up on a
 * bounded wait since the last call (its outputs are then incomplete), E_CUDA
 * on a CUDA error, else OK.
 */
cpattn_status cpattn_sync_status(cpattn_ctx* ctx, void* stream);

/*
 * Testing hook for the bounded-wait failure path.  flags = 1 makes one thread
 * of the first CTA of later cpattn_prefill launches skip one internal
 * arrival, so that CTA's waits expire after timeout_ms and it returns early;
 * cpattn_sync_status then reports E_TIMEOUT.  flags = 0 restores normal
 * operation.  timeout_ms <= 0 restores the default limit of 1000 ms per wait.
 */
cpattn_status cpattn_set_fault_injection(cpattn_ctx* ctx, int32_t flags, int32_t timeout_ms);

/*
 * Barrier accounting for tests (the PR's Design section: every signal must
 * be matched by its wait, or the kernel deadlocks).  Only the barrier-count
 * build of the library (compiled with -DCPATTN_COUNT_BARRIERS) implements
 * it; other builds return E_UNSUPPORTED.  Once `records` is registered, every
 * later prefill launch of this context adds, per CTA b (blockIdx), into
 * records[b * CPATTN_COUNT_RECORD ..] (uint32):
 *   row 0  [0, 40)    arrivals received by each mbarrier of CTA b (index =
 *                     the kernel's barrier number), from either CTA of a pair
 *   row 1  [40, 80)   completed waits of the softmax warps (one per warp)
 *   row 2  [80, 120)  completed waits of the TMA producer
 *   row 3  [120, 160) completed waits of the MMA warp
 *   row 4  [160, 200) softmax waits for the previous tile's P.V before a
 *                     rescale of O (data-dependent; apart from row 1)
 * The caller zeroes the records before a launch and reads them after it.
 * records: device memory, 4-byte aligned, at least (CTAs of the launch) *
 * CPATTN_COUNT_RECORD * 4 bytes (a launch has at most one CTA per SM), else
 * the prefill fails with E_INVALID; NULL turns counting off.
 * Errors: E_INVALID (NULL ctx, misaligned records), E_UNSUPPORTED.
 */
#define CPATTN_COUNT_BARS 40
#define CPATTN_COUNT_RECORD 200
cpattn_status cpattn_set_barrier_counts(cpattn_ctx* ctx, void* records, uint64_t bytes);

/*
 * Host-side view of the cache walk (no device work): for cache length L and
 * the context's P and S, writes the flat tile indices the prefill kernel
 * visits, in order, to tiles[0..n) and each tile's 128-column validity mask
 * as four 32-bit words to masks[4*i..4*i+4) (bit c of word c/32 set iff flat
 * row tile*128 + c of the (sequence, kv head) is a filled cache row).  *count
 * receives n; at most max_tiles entries are written (E_INVALID if more are
 * needed).  Either output pointer may be NULL to query the count only.
 */
cpattn_status cpattn_cache_walk(const cpattn_ctx* ctx, int32_t cache_len, int32_t* tiles,
                                uint32_t* masks, int32_t max_tiles, int32_t* count);

/*
 * The same view of the walk from its tile `first` on (first >= 0): the tiles
 * a split-KV piece that starts at virtual tile `first` visits, found by
 * skipping whole shard ranges as the kernel does.  Errors as above, and
 * E_INVALID for first < 0.
 */
cpattn_status cpattn_cache_walk_from(const cpattn_ctx* ctx, int32_t cache_len, int32_t first,
                                     int32_t* tiles, uint32_t* masks, int32_t max_tiles,
                                     int32_t* count);

/*
 * Allocation-free fused prefill.  The pages have no counterpart for this
 * entry point; it exists for callers that cannot allocate device memory --
 * code running while a pooled or custom allocator owns the device, regions
 * where cudaMalloc/cudaFree are forbidden or would synchronise (for example
 * while a stream is being captured), embedders that only pass pointers in.
 *
 * Same computation, arguments and layouts as cpattn_prefill, but it takes
 * the configuration directly instead of a context and never allocates: no
 * cudaMalloc, no cudaFree, no allocating library call, no host heap.  It
 * always runs the one-CTA-per-unit kernel form (cfg->pairing and
 * cfg->gqa_packing are checked but not used) and never splits a walk.  The
 * kernel's bounded-wait status word lives in a file-scope device array of
 * CPATTN_NOALLOC_SCRATCH_INTS ints (256 bytes) that every GPU loading the
 * library keeps until process exit.
 *  - The first call on a device resolves that array's device address and
 *    sets the kernel attributes for that device (with that device current);
 *    make that first call before any stream capture on the device.
 *  - Every call shares the array and clears the status word on `stream`
 *    before its launch.  Calls that overlap on the GPU (other streams, other
 *    threads) race on it; serialise them.
 *  - A device-side wait that expires still ends the kernel early (outputs
 *    incomplete) but is not reported by this call.
 *  - Sizes beyond the fixed host tables are refused: num_seqs >
 *    CPATTN_MAX_SEQS or more than CPATTN_MAX_ROW_BLOCKS row blocks return
 *    CPATTN_E_UNSUPPORTED, as do more than 64 devices.
 * Errors: E_INVALID (bad configuration or arguments, as for cpattn_create and
 * cpattn_prefill, or a buffer pointer the driver does not know as device or
 * managed memory), E_UNSUPPORTED (limits above), E_CUDA (set-up or launch).
 */
#define CPATTN_NOALLOC_SCRATCH_INTS 64
cpattn_status cpattn_prefill_noalloc(const cpattn_config* cfg, int32_t num_seqs,
                                     const int32_t* cache_lens, const int32_t* chunk_lens,
                                     const void* q, const void* k_new, const void* v_new,
                                     const void* k_cache, const void* v_cache, void* out,
                                     float* lse, void* stream);

/* Free the context (NULL-safe).  Does not synchronise. */
void cpattn_destroy(cpattn_ctx* ctx);

/* Static description of a status code. */
const char* cpattn_status_string(cpattn_status s);

/* Detail of the last error on this context (empty string if none). */
const char* cpattn_last_error(const cpattn_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H_ */
