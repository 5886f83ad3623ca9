// tma.cuh -- Tensor Memory Accelerator (cp.async.bulk.tensor) and mbarrier helpers.
//
// Tiles of activations are moved global -> shared by one elected thread with 3-D tensor
// copies that complete on an mbarrier; output tiles go shared -> global the same way.  Every
// wait is bounded: a wait that gives up reports failure to the caller, which records
// SSM_ERR_TIMEOUT in the status word, waits (bounded) for its own copies in flight and
// leaves.  Coordinates are always in range in dimension 0 (the box never starts outside the
// tensor there), so no copy starts at an unaligned or negative inner coordinate.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

constexpr uint32_t kSpinLimit = 1u << 22;  // try_wait polls before a wait is declared failed

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Make initialised barriers visible to the async proxy (the TMA unit) before first use.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async proxy (needed
// before a TMA store reads them).
__device__ __forceinline__ void fence_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

// Bounded wait for the phase with the given parity to complete.  Returns false on give-up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = smem_u32(bar);
  for (uint32_t i = 0; i < kSpinLimit; i++) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// 3-D tiled load (coordinates innermost first) completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// L2 eviction policy for the hinted copies below: evict_first, for data read or written for
// the last time (streamed tiles), so that it leaves L2 ahead of data that is read again.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// tma_load_3d with an L2 eviction policy.
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, int c0,
                                                 int c1, int c2, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)),
      "l"(pol)
      : "memory");
}

// 3-D tiled store from shared memory; elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0,
                                             int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(src))
      : "memory");
}

// tma_store_3d with an L2 eviction policy.
__device__ __forceinline__ void tma_store_3d_hint(const CUtensorMap* map, const void* src, int c0,
                                                  int c1, int c2, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group.L2::cache_hint "
      "[%0, {%1, %2, %3}], [%4], %5;" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(src)), "l"(pol)
      : "memory");
}

// A 4-byte global store with an L2 eviction policy.
__device__ __forceinline__ void st_global_hint(float* p, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}

// Drops the 128-byte L2 line at p (128-byte aligned) without writing it back: for scratch that is
// never read again, so that a dirty line costs no DRAM write.  The line's contents are undefined
// until it is written again.
__device__ __forceinline__ void discard_l2_line(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// Element index -> its place in a shared-memory box that a tensor map with a swizzle span of
// 16 << SWZ_B bytes (SWZ_B = 1, 2, 3: 32, 64, 128 bytes) fills or stores, for a buffer aligned
// to 1024 bytes: the 16-byte chunk index takes the XOR of address bits 7 .. 7 + SWZ_B - 1.
template <int SWZ_B, int ESIZE>
__device__ __forceinline__ int swizzled_index(int idx) {
  if constexpr (SWZ_B == 0) {
    return idx;
  } else {
    const int off = idx * ESIZE;
    return (off ^ (((off >> 7) & ((1 << SWZ_B) - 1)) << 4)) / ESIZE;
  }
}

__device__ __forceinline__ void tma_store_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until the committed stores no longer read their shared-memory source (<= n pending).
template <int N>
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until the committed stores are complete.
__device__ __forceinline__ void tma_store_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- host --------------------------------------------------------------------------------
// Encodes a 3-D tensor map over a row-major [d2][d1][d0] tensor (d0 fastest, element size
// `esize`, row stride `stride1` elements, plane stride `stride2` elements) with box
// {b0, b1, b2}.  `swizzle` = 32, 64 or 128 lays the box out in shared memory with that
// swizzle span (the 16-byte chunk index XOR address bits 7.. : see swizzled_index), 0 plainly.
// Returns false if the driver rejects it (alignment, box size).
bool encode_tmap_3d(CUtensorMap* map, const void* base, int esize, uint64_t d0, uint64_t d1,
                    uint64_t d2, uint64_t stride1, uint64_t stride2, uint32_t b0, uint32_t b1,
                    uint32_t b2, int swizzle = 0);

}  // namespace ssm
