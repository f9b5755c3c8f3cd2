// r4_device.cuh -- sm_103a device helpers: mbarriers with bounded waits, TMA,
// tcgen05 (tensor memory, MMA, copies, loads), shared-memory descriptors.
//
// Every wait on an mbarrier is bounded: after R4_WAIT_TIMEOUT_NS of global
// time it records an error code in the device error word, raises the CTA's
// abort flag and returns false, so a kernel whose copy or MMA never completes
// ends instead of hanging the GPU.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#ifndef R4_WAIT_TIMEOUT_NS
#define R4_WAIT_TIMEOUT_NS 2000000000ull  // 2 s of global time
// Upper bound on how long one mbarrier try_wait may suspend the thread (it
// resumes as soon as the phase completes): a waiting warp then issues no
// instructions instead of spinning against the warps doing the work.
#define R4_SUSPEND_HINT_NS 100000u
#endif

namespace r4 {

// Device error codes (written to the device error word).
enum : int {
  DEV_ERR_NONE = 0,
  DEV_ERR_WAIT_FULL = 1,     // consumer gave up waiting for a TMA stage
  DEV_ERR_WAIT_EMPTY = 2,    // producer gave up waiting for a free stage
  DEV_ERR_WAIT_ACC_FULL = 3, // epilogue gave up waiting for the accumulator
  DEV_ERR_WAIT_ACC_EMPTY = 4,// MMA issuer gave up waiting for the epilogue
  DEV_ERR_WAIT_DRAIN = 5,    // final drain of in-flight work gave up
  DEV_ERR_WAIT_PEER = 6      // split-K exchange gave up waiting for another CTA of the cluster
};

// Split-K arrival counters (one int per output tile in the caller's
// workspace): every unit of a tile adds 1 when its partial is written; the
// last of the tile's `splits` arrivals sums the partials and resets the
// counter to 0. A launch that stopped early (an expired wait) still arrives,
// for every unit it owed, with kPoisonArrival added: the last arrival then
// skips the sum (its partials are incomplete) but still resets the counter,
// so the workspace is zero again for the next call either way.
constexpr int kArrivalMask = 0xFFFF;      // arrivals (splits <= 64)
constexpr int kPoisonShift = 16;
constexpr int kPoisonArrival = 1 << kPoisonShift;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31; }

__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(pred));
  return pred != 0;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(R4_SUSPEND_HINT_NS)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase with the given parity (no suspension).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete. Returns false
// (and raises *abort, records `code` in *err) on timeout, or false at once if
// another role of the CTA has already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          int *err, int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > R4_WAIT_TIMEOUT_NS) {
        *abort = 1;
        atomicCAS(err, 0, code);   // keep the first error recorded
        return false;
      }
    }
  }
}

// mbar_wait by spinning on test_wait instead of a suspending try_wait, same
// bounds and error contract. For handshakes on the critical path of every
// K block, where waking a suspended thread costs more than the spin (block-
// FP8 promotion on GB300: 3-4 % faster).
__device__ __forceinline__ bool mbar_spin_wait(uint64_t *bar, uint32_t parity, volatile int *abort, int *err,
                                               int code) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > R4_WAIT_TIMEOUT_NS) {
        *abort = 1;
        atomicCAS(err, 0, code);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------- TMA

// ---------------------------------------------------------------- thread-block clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// Arrive on an mbarrier of another CTA of the cluster (address from
// mapa_shared); release at cluster scope orders this thread's earlier
// writes (and what it synchronised with) before the arrival.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(R4_SUSPEND_HINT_NS)
      : "memory");
  return ok != 0;
}

// Bounded wait with cluster-scope acquire (the phase was completed by
// arrivals from other CTAs of the cluster); same contract as mbar_wait.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, volatile int *abort, int *err,
                                                  int code) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > R4_WAIT_TIMEOUT_NS) {
        *abort = 1;
        atomicCAS(err, 0, code);
        return false;
      }
    }
  }
}

__device__ __forceinline__ float4 ld_dsmem_f32x4(uint32_t cluster_addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(cluster_addr)
               : "memory");
  return v;
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t cluster_addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
  return v;
}

__device__ __forceinline__ void fence_acq_rel_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }

// Split cluster barrier (every thread of every CTA): arrive releases this
// thread's earlier accesses; wait returns once every thread of the cluster
// has arrived.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Full cluster barrier, executed by every thread of every CTA of the cluster.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Warp-wide bounded wait: lane 0 polls the barrier (an mbarrier poll by all
// 32 lanes is 32 shared-memory barrier operations), the warp then syncs and
// every lane gets lane 0's result. The warp barrier orders the lanes'
// following accesses after lane 0's acquire.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort, int *err,
                                          int code) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort, err, code);
  __syncwarp();
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// warp_wait with lane 0 spinning (mbar_spin_wait).
__device__ __forceinline__ bool warp_spin_wait(uint64_t *bar, uint32_t parity, volatile int *abort, int *err,
                                               int code) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_spin_wait(bar, parity, abort, err, code);
  __syncwarp();
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *m, uint64_t *bar, int x, int y,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *m, uint64_t *bar, int x, int y,
                                            int z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "l"(policy)
      : "memory");
}

// Plain bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Bulk prefetch of [src, src + bytes) from global memory into L2 (no smem).
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMA tensor store of a 2-D box from shared memory (bulk-group completion),
// and the bulk-group commit / waits of the issuing thread.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *m, const void *src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(x), "r"(y), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive (once) on `bar` when all tcgen05 operations issued so far by this
// thread have completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Shared -> tensor memory copy: 32 rows x 16 bytes, replicated into all four
// 32-lane quarters of tensor memory (4 columns).
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// D[tmem] (+)= A[smem] x B[smem]^T with ue8m0 block scales from tensor memory,
// one scale per 32 K (kind::mxf8f6f4, M=128, K=32 per instruction).
__device__ __forceinline__ void tc_mma_mxf8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}\n" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[smem] x B[smem]^T with packed e2m1 operands (two per byte)
// and ue8m0 block scales from tensor memory, one scale per 32 K: kind::mxf4,
// M = 128, K = 64 per instruction, scale_vec::2X (scale id 0 or 2 selects the
// byte pair of each row's 32-bit scale column).
__device__ __forceinline__ void tc_mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}\n" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[smem] x B[smem]^T, fp8/fp6/fp4 operands without block scale.
__device__ __forceinline__ void tc_mma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (quarter*32 + i), columns [col, col+32).
__device__ __forceinline__ void tc_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tc_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns into a 16-register array.
__device__ __forceinline__ void tc_ld_32x32b_x16h(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// 16 lanes x 32 consecutive 32-bit columns in the 16x256b shape (four
// 8-column repeats), into r[0..16). Thread i of the warp receives, in repeat
// g (registers 4g..4g+3): lane i/4 at columns 8g + 2(i%4) and 8g + 2(i%4) + 1,
// then lane 8 + i/4 at the same two columns -- the accumulator fragment of
// the warp-level m16n8 MMA, which is the fragment stmatrix consumes. (Checked
// on GB300: an epilogue built on this reading reproduces the 32x32b one bit
// for bit.)
__device__ __forceinline__ void tc_ld_16x256b_x4(uint32_t taddr, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Two floats to a bf16 pair (round to nearest even): lo in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Four 8x8 b16 matrices to shared memory, transposed: register k of thread i
// holds row i/4, columns 2(i%4) and 2(i%4) + 1 of matrix k; thread 8k + j
// supplies the 16-byte-aligned address at which column j of matrix k is
// stored as 8 consecutive b16.
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}

// ---------------------------------------------------------------- descriptors

// Shared-memory matrix descriptor, K-major operand in the 128-byte swizzle
// layout: rows of 128 bytes, 8-row groups 1024 bytes apart (SBO), tile base
// 1024-byte aligned. Selecting a K slice inside the 128-byte row is done by
// adding its byte offset to the start address.
__device__ __forceinline__ uint64_t sdesc_sw128_kmajor(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;                 // LBO (unused for swizzled K-major)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;         // SBO: 8 rows x 128 B
  d |= static_cast<uint64_t>(1u) << 46;                 // descriptor version (tcgen05)
  d |= static_cast<uint64_t>(2u) << 61;                 // 128-byte swizzle
  return d;
}

// Descriptor for a 32-row x 16-byte scale-factor block (no swizzle, rows 16 B
// apart, 8-row core matrices 128 B apart), the source of tcgen05.cp 32x128b.
__device__ __forceinline__ uint64_t sdesc_sf_32x16(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(128u >> 4) << 32;          // SBO: 8 rows x 16 B
  d |= static_cast<uint64_t>(1u) << 46;
  return d;
}

// Instruction descriptor, kind::mxf8f6f4 with ue8m0 block scales:
// A = e2m1 (format 5), B = e4m3 (format 0), both K-major, M = 128.
__host__ __device__ constexpr uint32_t idesc_mxf8f6f4_e2m1_e4m3(int n, int a_sf_id, int b_sf_id) {
  return (static_cast<uint32_t>(b_sf_id & 3) << 4) | (5u << 7) | (0u << 10) |
         (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(128 >> 4) << 24) |
         (static_cast<uint32_t>(a_sf_id & 3) << 29);
}

// Instruction descriptor, kind::f8f6f4: A = B = e4m3, fp32 accumulate,
// K-major, M = 128.
__host__ __device__ constexpr uint32_t idesc_f8f6f4_e4m3(int n) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(128 >> 4) << 24);
}

// ---------------------------------------------------------------- programmatic dependent launch
// Kernels are launched with programmatic stream serialization: the next
// kernel in the stream may start while this one runs. Each kernel reads
// data that does not depend on earlier kernels (weights) before pdl_wait(),
// and touches everything else (activations, scales, outputs, workspace) only
// after it. pdl_wait() returns once the preceding grid has completed and its
// memory is visible; without a programmatic predecessor it returns at once.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- misc

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Barrier over `nthreads` threads that also ORs a per-thread flag: every
// participant gets the same result (used to agree on stopping).
__device__ __forceinline__ bool named_bar_any(int id, int nthreads, bool flag) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"(flag ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return out != 0;
}

// Two fp32 fused multiply-adds in one instruction: (d0, d1) += (a0, a1) * (b0, b1),
// each rounded once (IEEE fma).
__device__ __forceinline__ void fma_f32x2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rc;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%0, %1};\n\tfma.rn.f32x2 rc, ra, rb, rc;\n\tmov.b64 {%0, %1}, rc;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Two fp32 multiplies in one instruction: (d0, d1) *= (a0, a1), each rounded once.
__device__ __forceinline__ void mul_f32x2(float &d0, float &d1, float a0, float a1) {
  asm("{\n\t.reg .b64 ra, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rd, {%0, %1};\n\t"
      "mul.rn.f32x2 rd, rd, ra;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1));
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float v) {
  __nv_bfloat16 h = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t *>(&h);
}

// Split-K epilogue of the last-arriving CTA: sum `nslots` fp32 partial tiles
// (each [tokens][128 n], n contiguous; slot(s) is the s-th) in s order --
// deterministic -- and store bf16(scale[t] * sum) (scale == nullptr: 1) into
// C[t0 + t][n0 + n] for t < tmax, n0 + n < N. The loads are independent L2
// reads (.cg: the partials were written by other SMs), four n per thread.
template <int U = 4, int S = 4, class SlotFn>
__device__ __forceinline__ void reduce_slots_store(SlotFn slot, int nslots, int tmax, int n0, int N,
                                                   const float *scale, int t0, uint16_t *c, int ldc, int tid,
                                                   int nthreads) {
  // Each pass covers U float4 groups per thread and keeps up to U x S loads
  // in flight (S slots at a time), so the pass costs about one L2 round trip
  // per S slots instead of one per slot and group. (Kernels under a tight
  // register cap take smaller U and S.)
  const int total = tmax * 32;
  for (int base = tid; base < total; base += nthreads * U) {
    float4 acc[U];
    const float *s0 = slot(0);
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int idx = base + k * nthreads;
      acc[k] = idx < total ? __ldcg(reinterpret_cast<const float4 *>(s0 + (idx >> 5) * 128 + (idx & 31) * 4))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int s2 = 1; s2 < nslots; s2 += S) {
      float4 v[S][U];
#pragma unroll
      for (int ss = 0; ss < S; ++ss) {
        const float *sp = s2 + ss < nslots ? slot(s2 + ss) : nullptr;
#pragma unroll
        for (int k = 0; k < U; ++k) {
          const int idx = base + k * nthreads;
          v[ss][k] = (sp != nullptr && idx < total)
                         ? __ldcg(reinterpret_cast<const float4 *>(sp + (idx >> 5) * 128 + (idx & 31) * 4))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int ss = 0; ss < S; ++ss)   // in slot order (deterministic)
        if (s2 + ss < nslots) {
#pragma unroll
          for (int k = 0; k < U; ++k) {
            acc[k].x += v[ss][k].x;
            acc[k].y += v[ss][k].y;
            acc[k].z += v[ss][k].z;
            acc[k].w += v[ss][k].w;
          }
        }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int idx = base + k * nthreads;
      if (idx >= total) continue;
      const int tl = idx >> 5, n4 = (idx & 31) * 4;
      const float sc = scale ? __ldg(scale + t0 + tl) : 1.f;
      const int n = n0 + n4;
      uint16_t *dst = c + static_cast<size_t>(t0 + tl) * ldc + n;
      const float vals[4] = {acc[k].x * sc, acc[k].y * sc, acc[k].z * sc, acc[k].w * sc};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (n + j < N) dst[j] = f32_to_bf16_rn(vals[j]);
    }
  }
}

// The same for `splits` partial tiles [BT][128] stored one after another.
template <int BT, int U = 4, int S = 4>
__device__ __forceinline__ void reduce_partials_store(const float *base, int splits, int tmax, int n0, int N,
                                                      const float *scale, int t0, uint16_t *c, int ldc, int tid,
                                                      int nthreads) {
  constexpr size_t kTile = 128 * BT;
  reduce_slots_store<U, S>([&](int s2) { return base + s2 * kTile; }, splits, tmax, n0, N, scale, t0, c, ldc, tid,
                           nthreads);
}

}  // namespace r4
