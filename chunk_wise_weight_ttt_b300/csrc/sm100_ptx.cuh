// Inline-PTX building blocks for sm_100-family (sm_103a) kernels: mbarriers
// (local and across a CTA pair of a cluster), TMA tensor loads into one CTA's
// own shared memory (no multicast loads), TMA tensor stores from it, L2
// prefetches, and the
// 5th-generation tensor core in its CTA-pair form (tcgen05 cta_group::2: TMEM
// allocation, MMA issue, commit, TMEM loads).  Every mbarrier wait here is
// bounded by wall-clock time so that no kernel can hang the GPU.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace ttt {

// Longest a single in-kernel wait may last before it gives up (nanoseconds).
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Error codes written to the workspace's error word.
enum : int {
  kErrNone = 0,
  kErrWaitTmaFull = 1,
  kErrWaitSmemEmpty = 2,
  kErrWaitAccFull = 3,
  kErrWaitAccEmpty = 4,
  kErrWaitSched = 5,
  kErrWaitDrain = 6,
  kErrWaitDep = 7,
  kErrWaitEpi = 8,
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the barrier's phase with the given parity has completed.
// Returns false if the CTA-wide abort flag is raised or the time limit runs
// out (in which case the abort flag is raised and `code` is recorded).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int* err_word, int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicCAS(err_word, 0, code);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------- cross-CTA dependencies

// Release-add to a global counter (after this thread's earlier writes).
__device__ __forceinline__ void dep_signal(int* counter, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(counter), "r"(v) : "memory");
}

__device__ __forceinline__ int dep_load(const int* counter) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
  return v;
}

// Order this thread's generic-proxy global accesses with its later (or
// earlier) async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Wait until *counter >= target (acquire).  Bounded like mbar_wait: gives up
// when the CTA's abort flag is raised or after kWaitLimitNs (raising it and
// recording `code`).
__device__ __forceinline__ bool dep_wait(const int* counter, int target, volatile int* abort_flag,
                                         int* err_word, int code) {
  if (dep_load(counter) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    __nanosleep(64);
    if (dep_load(counter) >= target) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicCAS(err_word, 0, code);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------- cluster

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address in the shared memory of CTA `rank` of this cluster that corresponds
// to the local shared-memory address `local` (a shared::cluster address).
__device__ __forceinline__ uint32_t cluster_map(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Arrive (release at cluster scope) on an mbarrier given by its shared::cluster
// address, which may lie in another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// All threads of every CTA of the cluster.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// ---------------------------------------------------------------- programmatic dependent launch

// Block until every grid this one depends on has completed and its memory is
// visible (returns at once when the grid was launched without a dependency).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next dependent grid on the stream to be scheduled (its CTAs still
// wait in griddep_wait for this grid to complete).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Load of one box into this CTA's shared memory whose completion (transaction
// bytes) is signalled on an mbarrier that may lie in the peer CTA of a CTA pair
// (`bar_cluster` is a shared::cluster address, e.g. from cluster_map).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster)
      : "memory");
}

// Prefetch one box of a tensor map into L2 (no shared memory is written and
// nothing is signalled); coordinates as for tma_load_2d.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1)
               : "memory");
}

// Store of one box from this CTA's shared memory (laid out as a load through
// the same map would lay it out) to global memory, as part of the issuing
// thread's current bulk group.  Elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* smem_src, int32_t c0,
                                             int32_t c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(smem_src)), "r"(c0), "r"(c1)
               : "memory");
}

// Close the issuing thread's current bulk group of TMA stores.
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Block until at most N of this thread's committed bulk groups are still
// reading their shared-memory sources (their buffers may then be rewritten).
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Block until at most N of this thread's committed bulk groups are incomplete
// (the others' global writes are done).
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
//
// The engine pairs two CTAs on one MMA, so every tcgen05 instruction here is
// the cta_group::2 form (allocation, MMA, commit).

// cta_group::2: one warp of each CTA of the pair performs these together; the
// same columns are allocated in both CTAs' TMEM.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
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

// Pair MMA (cta_group::2), issued by one thread of the even CTA: A rows
// [0, M/2) and B rows [0, N/2) come from this CTA's shared memory, the other
// halves from the same offsets in the peer's; each CTA's TMEM receives its
// M/2 accumulator rows.
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}


// Pair forms of the commits: arrive once on `bar` in this CTA, or at `bar`'s
// offset in every CTA of `cta_mask`, when the pair's tcgen05 ops issued so
// far by this thread are done.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_commit_pair_mc(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}


// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulation.
// Field layout: [4,6) D format (1 = f32), [7,10) A format (1 = bf16),
// [10,13) B format (1 = bf16), bit 15 A major (1 = MN-major), bit 16 B major,
// [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.  Fields: [0,14) start
// address >> 4, [16,30) leading byte offset >> 4, [32,46) stride byte offset
// >> 4, [46,48) descriptor version (1), [61,64) layout (2 = 128B swizzle).
// K-major operand (rows of 128 B along K, 8-row groups 1024 B apart):
//   lbo unused, sbo = 1024.
// MN-major operand (rows of 128 B = 64 bf16 along M/N, one row per K index,
//   64-element M/N blocks `lbo` bytes apart, 8-row K groups `sbo` = 1024 apart).
// The constant (address-free) part of such a descriptor: the descriptor for
// shared-memory address `a` is this value | ((a & 0x3FFFF) >> 4), and
// advancing the address by `off` bytes adds off >> 4 (the operands lie below
// 2^18, so the 14-bit start field never carries).
__host__ __device__ constexpr uint64_t sdesc_sw128_hi(uint32_t lbo, uint32_t sbo) {
  return (static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16) |
         (static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// 32 lanes x 32 consecutive fp32 columns: thread i of the warp gets lane
// (base lane + i), columns [col, col+32).  The registers are only valid after
// tmem_ld_wait(), which takes them as operands so no use is hoisted above it.
#define TTT_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                  "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define TTT_P8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), \
                  "+r"(r[i + 4]), "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : TTT_R8(0), TTT_R8(8), TTT_R8(16), TTT_R8(24)
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : TTT_P8(0), TTT_P8(8), TTT_P8(16), TTT_P8(24)::"memory");
}

#undef TTT_R8
#undef TTT_P8

}  // namespace ttt
