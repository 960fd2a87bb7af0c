// ptx.cuh -- inline-PTX helpers for sm_103a: mbarrier, TMA bulk tensor
// copies, the global timer.  Every wait here has a time limit so that a
// pipeline that never fills returns an error instead of hanging the GPU.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace sgemm {
namespace ptx {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the other threads and to the
// async (TMA) proxy before first use.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Non-blocking probe of a phase (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Shared-memory fetch-and-add with acquire-release semantics at CTA scope:
// this thread's earlier accesses are ordered before the add, and the adds
// of other threads that precede it in the counter's order are visible
// after it.
__device__ __forceinline__ unsigned int atom_add_acq_rel_cta(unsigned int* addr, unsigned int v) {
  unsigned int old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(smem_addr(addr)), "r"(v)
               : "memory");
  return old;
}

// Flag handshake between CTAs of one grid (stream-K partial tiles): the
// writer releases after its data stores, the reader acquires before its loads.
__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(unsigned int* p, unsigned int v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait until the phase with the given parity of barrier `bar` completes.
// Returns false if it has not completed after timeout_ns nanoseconds.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
#pragma unroll 1
  for (int i = 0; i < 64; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

// As mbar_wait, but also gives up as soon as *abort (a flag the CTA's other
// roles set when one of them fails) is non-zero.
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                                   const volatile int* abort) {
#pragma unroll 1
  for (int i = 0; i < 64; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort || globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

// After a failed wait, before the CTA exits: wait (bounded) until the
// copies of the last `stages` slices issued into a ring have landed, so no
// copy writes shared memory that a later CTA owns.  Slice j used stage
// j % stages (its full barrier at bar_full + stride * stage) in phase
// j / stages; every earlier slice was waited on before its stage was reused.
// Each wait lasts at least 100 ms, however short the configured limit, which
// is far above a copy's latency.
__device__ __forceinline__ void drain_ring(uint32_t bar_full, uint32_t stride, uint32_t issued, uint32_t stages,
                                           uint64_t timeout_ns) {
  const uint64_t limit = timeout_ns < 100000000ull ? 100000000ull : timeout_ns;
#pragma unroll 1
  for (uint32_t j = issued > stages ? issued - stages : 0u; j < issued; ++j)
    mbar_wait(bar_full + stride * (j % stages), (j / stages) & 1u, limit);
}

// drain_ring for a ring refilled by "the warp that completes a stage's
// release set": released[s] counts the warp releases of stage s, and the
// release set of slice j (every `warps`-th release) issued slice
// j + stages when that is below `total`.  So stage s received one copy in
// the prologue (s < total) plus one per completed set, up to the number of
// slices j = s (mod stages) with j + stages < total; the last of them is the
// only one that can be in flight.
__device__ __forceinline__ void drain_ring_released(uint32_t bar_full, uint32_t stride, const unsigned int* released,
                                                    uint32_t warps, uint32_t stages, uint32_t total,
                                                    uint64_t timeout_ns) {
  const uint64_t limit = timeout_ns < 100000000ull ? 100000000ull : timeout_ns;
#pragma unroll 1
  for (uint32_t s = 0; s < stages && s < total; ++s) {
    const uint32_t sets = *reinterpret_cast<const volatile unsigned int*>(released + s) / warps;
    const uint32_t refills = (total - 1u - s) / stages;
    const uint32_t copies = 1u + (sets < refills ? sets : refills);
    mbar_wait(bar_full + stride * s, (copies - 1u) & 1u, limit);
  }
}

// 2-D tiled TMA load of the box at (x = inner coordinate, y = outer) into
// shared memory at `dst`; completion is signalled on `bar` as transaction
// bytes.  x * 4 bytes must be a multiple of 16 (callers pass multiples of 4).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 3-D tiled TMA load: (x, y) as tma_load_2d, z the outermost coordinate
// (the batch index of a strided batch).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// As tma_load_2d, with an L2 eviction-priority hint (a policy made by
// l2_policy_evict_first / l2_policy_evict_last).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// As tma_load_3d, with an L2 eviction-priority hint.
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// L2 policy: data read once (stream it through, evict first).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// L2 policy: data reused by many CTAs (keep it).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ float4 lds128(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

}  // namespace ptx
}  // namespace sgemm
