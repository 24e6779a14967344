// Asynchronous shared-memory copies for the libtq kernels (sm_103a): mbarrier
// wrappers, 2-D tensor copies (cp.async.bulk.tensor), an L2 eviction policy for
// data read once, the programmatic-dependent-launch wait, and a bounded mbarrier
// wait that gives up after about a second instead of spinning forever.
#pragma once

#include <cuda.h>  // CUtensorMap (the type only; no driver calls here)
#include <stdint.h>

namespace tq {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// L2 policy for data read once per call (the decode's pages): evicted first, so
// the small data every call re-reads (block tables, context lengths, queries,
// split partials) stays in L2 while gigabytes of pages stream through it.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Waits for the grid this one was launched as a programmatic dependent of (no-op
// for an ordinary launch).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_try(uint32_t addr, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(addr), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait on an mbarrier phase: gives up after ~1 s (returns false).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try(addr, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try(addr, parity)) return true;
    if ((it & 63) == 63 && global_ns() - t0 > 1000000000ull) return false;
  }
  return false;
}

// 2-D tiled copy of one box of `tmap` at element coordinates (c0 inner, c1 outer)
// into shared memory at `dst` (a shared-space address), completing on `bar`.
__device__ __forceinline__ void tensor_copy_2d(uint32_t dst, const CUtensorMap* tmap, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// Orders this thread's earlier shared-memory accesses (and those it has seen
// through a warp or CTA barrier) before its later asynchronous-proxy copies.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

}  // namespace tq
