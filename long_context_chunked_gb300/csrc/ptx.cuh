// Thin inline-PTX wrappers for sm_103a: mbarrier, TMA tensor loads and the
// 5th-generation tensor-core (tcgen05) instructions with TMEM accumulators.
// Every wait in this library is bounded; see BoundedWait below.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace cpattn {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrivals on an mbarrier of another CTA of the cluster (shared::cluster
// address from mapa_shared).  They keep the default release.cta semantics:
// what crosses a CTA pair through these barriers is TMEM contents (ordered
// by the tcgen05 fences around the barrier operations) and TMA data
// (ordered by the transaction count), never generic-proxy stores -- and a
// cluster-scope release costs each arrival a long fence.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx_remote(uint32_t bar_cluster,
                                                             uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cluster.b64 _, [%0], %1;" ::"r"(bar_cluster),
               "r"(bytes)
               : "memory");
}

// Device status word codes (written by the first role that gives up).
enum : int { kStatusOk = 0, kStatusTimeout = 1, kStatusLayout = 2, kStatusRange = 3 };

// ------------------------------------------------------ barrier-count build
// Built with -DCPATTN_COUNT_BARRIERS, the prefill kernels count every
// mbarrier arrival and every completed wait into a caller-owned record per
// CTA (kCountRecord uint32 each, indexed by blockIdx.x): row 0 holds the
// arrivals each barrier of this CTA received (from either CTA of a pair),
// rows 1-3 the waits completed by the softmax warps, the producer and the MMA
// warp (one per warp and completed wait), row 4 the softmax waits for the
// previous tile's P.V that precede a rescale of O.  A test checks at kernel
// exit that every barrier's arrivals form whole phases and that every
// waiter observed every phase it consumes.  In other builds these helpers
// are empty and compile away.
constexpr int kCountBars = 40;
constexpr int kCountRowArrive = 0, kCountRowSoftmax = 1, kCountRowProducer = 2,
              kCountRowMma = 3, kCountRowRescale = 4;
constexpr int kCountRecord = 5 * kCountBars;

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// n arrivals on barrier `bar` of every CTA of the cluster whose rank is set
// in cta_mask (bit 0: rank 0; a plain launch is a cluster of one).
__device__ __forceinline__ void count_arrive(uint32_t* counts, uint32_t cta_mask, int bar,
                                             uint32_t n) {
#ifdef CPATTN_COUNT_BARRIERS
  if (counts == nullptr) return;
  const uint32_t first = blockIdx.x - cluster_ctarank();
  for (uint32_t r = 0; r < 2; ++r)
    if (cta_mask & (1u << r)) atomicAdd(counts + (first + r) * kCountRecord + bar, n);
#else
  (void)counts, (void)cta_mask, (void)bar, (void)n;
#endif
}

// The same for a warp-collective arrival (a tcgen05.commit that one elected
// lane of a converged warp issues): counted once, by lane 0.
__device__ __forceinline__ void count_commit(uint32_t* counts, uint32_t cta_mask, int bar) {
  if ((threadIdx.x & 31) == 0) count_arrive(counts, cta_mask, bar, 1);
}

// One completed wait on barrier `bar` of this CTA, by the role of `row`.
__device__ __forceinline__ void count_wait(uint32_t* counts, int row, int bar) {
#ifdef CPATTN_COUNT_BARRIERS
  if (counts != nullptr && (threadIdx.x & 31) == 0)
    atomicAdd(counts + blockIdx.x * kCountRecord + row * kCountBars + bar, 1u);
#else
  (void)counts, (void)row, (void)bar;
#endif
}

// A wait with a wall-clock limit.  On expiry it records the site in the
// device status word, raises the CTA-wide abort flag and returns false; a
// wait also returns false as soon as another role of the CTA has aborted,
// so one expired wait ends every role's loop promptly instead of hanging.
struct BoundedWait {
  volatile int* abort_flag;  // shared memory
  int* status;               // global status word (may be null)
  uint64_t limit_ns;
  uint32_t* counts;          // barrier-count build: the records, else unused
  uint32_t bar0;             // shared address of barrier 0 (count index base)
  int row;                   // count row of the waiting role

  __device__ __forceinline__ BoundedWait with_row(int r) const {
    BoundedWait w = *this;
    w.row = r;
    return w;
  }

  __device__ __forceinline__ bool operator()(uint32_t bar, uint32_t parity, int site) const {
    if (mbar_try_wait(bar, parity)) return done(bar);
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
      for (int i = 0; i < 32; ++i)
        if (mbar_try_wait(bar, parity)) return done(bar);
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        if (status != nullptr) atomicCAS(status, kStatusOk, (site << 8) | kStatusTimeout);
        return false;
      }
    }
  }

 private:
  __device__ __forceinline__ bool done(uint32_t bar) const {
    count_wait(counts, row, static_cast<int>((bar - bar0) >> 3));
    return true;
  }
};

// Wait that ignores the abort flag: used only to let copies and MMAs that are
// already in flight land before a CTA that gave up leaves the kernel.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > limit_ns) return false;
  return true;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before the kernel ahead of it on the stream has
// finished; griddep_wait blocks the calling thread until that grid has
// completed and its writes are visible (immediately, when the launch was an
// ordinary one).  griddep_launch_dependents lets the next kernel start once
// every block of this grid has called it or exited.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Register reallocation between warpgroups (every warp of a warpgroup
// executes the same one): .inc waits until the CTA's pool, which the launch
// sized at threads x registers per thread, has that many free per thread --
// the other warpgroups' .dec must free them, so the shares of all
// warpgroups may not add up to more than the launch allocation.
template <int N>
__device__ __forceinline__ void reg_alloc_inc() {
  static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg operand");
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void reg_alloc_dec() {
  static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg operand");
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads.
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t count, bool pred) {
  uint32_t res;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(res)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
      : "memory");
  return res != 0;
}

// --------------------------------------------------------------- TMA loads
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 3-D tiled load of one box into shared memory, completing `bytes` of
// transaction count on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// Load for a CTA pair running 2-SM MMAs: the box lands in THIS CTA's shared
// memory at dst, and its transaction bytes complete on the mbarrier at
// bar_cluster -- the leader CTA's barrier (mapa_shared(bar, 0)), which is
// the one the leader's MMA thread waits on.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* m,
                                                 uint32_t bar_cluster, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2 [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(bar_cluster)
      : "memory");
}

// Whole-cluster barrier (every thread of every CTA of the cluster).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ----------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Paired-SM (cta_group::2) allocation: executed by one warp of EACH CTA of
// the pair; both receive the same TMEM address, and the leader's 2-SM MMAs
// address both CTAs' TMEM through it.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// MMA issue and commit are WARP-COLLECTIVE here: every lane of a converged
// warp executes the call with the same operands, and the one lane that
// elect.sync picks issues the instruction.  With all 32 lanes active it
// elects the same (lowest) lane every time, so every MMA and commit of a
// role comes from one thread: the MMAs execute in issue order and each
// commit tracks all of them.  Issuing from a whole warp keeps
// the operands warp-uniform; a lone lane in a divergent branch issues more
// slowly when the softmax warps on its SM sub-partition use most issue slots
// (measured: 1852 vs 1537 clocks for 24 MMAs of 64 clocks each).

// D[tmem] (+)= A[smem] * B[smem], kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem].
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 2-SM MMAs, issued by the leader CTA of a pair: M = 256 rows, rows 0-127
// in the leader's TMEM lanes and A (shared memory or TMEM), rows 128-255 in
// the peer's, at the same addresses; B is split by N, each CTA holding N/2
// columns of it at the same shared-memory offset.
__device__ __forceinline__ void mma2_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma2_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Completion of the leader's 2-SM MMAs, signalled on the mbarrier at the
// same offset in every CTA of cta_mask.
__device__ __forceinline__ void mma2_commit_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n\t}" ::"r"(bar), "h"(cta_mask)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by the
// issuing thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// tcgen05.ld, 32x32b shape: thread i of the warp reads TMEM lane (the warp's
// lane quarter) + i, 32 consecutive fp32 columns starting at taddr's column.
// The wait::ld sits in the same asm statement, so the outputs are valid when
// it returns (with a separate wait the compiler could read them too early).
__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// The same load without the wait: the registers must not be read before
// tmem_ld32_fence() on the same array.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Wait for this thread's outstanding TMEM loads; the registers pass through
// the asm as read-write operands so no use of them can move above the wait.
__device__ __forceinline__ void tmem_ld32_fence(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, M x N tile;
// b_mn_major selects an N-contiguous B operand (the V tile of P.V).
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4)                                  // D format: fp32
         | (1u << 7)                                // A format: bf16
         | (1u << 10)                               // B format: bf16
         | ((b_mn_major ? 1u : 0u) << 16)           // B major-ness
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}
// The same with A and B in fp16 (format code 0).
__host__ __device__ constexpr uint32_t make_idesc_f16(int M, int N, bool b_mn_major) {
  return (1u << 4)                                  // D format: fp32
         | ((b_mn_major ? 1u : 0u) << 16)           // B major-ness
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand: start
// address, leading- and stride-dimension byte offsets (both /16), the
// descriptor version bit and the 128B swizzle mode.
__device__ __forceinline__ uint64_t make_sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                     uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  // cvt packs its first source into the upper half.
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two fp32 values rounded to nearest-even fp16, lo in the lower half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight bf16 values (one 16-byte vector) as eight fp16 values, rounded to
// nearest-even (bf16 -> fp32 is exact); *overflow is set when a result is
// infinite or NaN, i.e. the value lies outside fp16's finite range.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v, bool* overflow) {
  auto conv = [&](uint32_t w) {
    const uint32_t h = pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    // exponent field all ones in either half: inf or NaN
    if ((h & 0x7C00u) == 0x7C00u || (h & 0x7C000000u) == 0x7C000000u) *overflow = true;
    return h;
  };
  return make_uint4(conv(v.x), conv(v.y), conv(v.z), conv(v.w));
}

}  // namespace cpattn
