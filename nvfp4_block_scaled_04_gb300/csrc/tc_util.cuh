// mbarrier, TMA and bulk-copy helpers shared by the TMA-fed kernels
// (sm_103a). Every wait is bounded by the global timer: a wait that gives up
// records NVFP4_ERR_TIMEOUT in the device status word it is handed, raises
// the caller's CTA-local abort flag and returns false, so no kernel spins
// forever.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace nvfp4 {

constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;  // 2 s

NVFP4_DEV uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

NVFP4_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

NVFP4_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

// Wait for `parity` on `bar`; give up after limit_ns, or as soon as another
// role of the CTA has given up. Returns false on give-up.
NVFP4_DEV bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status,
                                 unsigned long long limit_ns = WAIT_LIMIT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t n = 0;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63) == 63) {
      if (abort_flag && *abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) {
        if (status) atomicExch(status, NVFP4_ERR_TIMEOUT);
        if (abort_flag) *abort_flag = 1;
        return false;
      }
    }
  }
}

// ---- barriers that threads or the tensor cores of the other CTA of a
// cluster arrive on (CTA pairs)

NVFP4_DEV bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait (cluster-scope acquire), with the give-up rules of mbar_wait_bounded.
NVFP4_DEV bool mbar_wait_cluster_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t n = 0;; ++n) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((n & 63) == 63) {
      if (abort_flag && *abort_flag) return false;
      if (globaltimer() - t0 > WAIT_LIMIT_NS) {
        if (status) atomicExch(status, NVFP4_ERR_TIMEOUT);
        if (abort_flag) *abort_flag = 1;
        return false;
      }
    }
  }
}

// Arrive on the barrier at the same shared-memory offset in CTA `rank` of the cluster.
NVFP4_DEV void mbar_arrive_cluster(uint32_t bar, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(bar), "r"(rank));
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}

// Arrive once on the barrier at this offset in both CTAs of the pair when the
// tensor-core operations this thread issued so far have completed.
NVFP4_DEV void tc_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

NVFP4_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

NVFP4_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

NVFP4_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

NVFP4_DEV void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Four rows r0..r3 of a 2-D tensor map whose box is one row high, starting at
// column x, into consecutive box-sized slots at dst.
NVFP4_DEV void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int r0, int r1, int r2, int r3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(map), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
      : "memory");
}

NVFP4_DEV void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// L2 eviction priority for data a kernel reads exactly once (streamed
// weights): evict_first keeps it from displacing what L2 holds for others.
NVFP4_DEV uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// tma_load_2d with an L2 cache policy (from createpolicy).
NVFP4_DEV void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start >> 4 at bit 0, leading
// byte offset >> 4 at bit 16, stride byte offset >> 4 at bit 32, version 1
// at bit 46, layout (swizzle mode) at bit 61.
NVFP4_DEV uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  return (uint64_t((addr & 0x3FFFFu) >> 4)) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (uint64_t(layout) << 61);
}

// Programmatic dependent launch: let the next kernel on the stream start
// early / wait here until the previous kernel's results are visible.
NVFP4_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
NVFP4_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace nvfp4
