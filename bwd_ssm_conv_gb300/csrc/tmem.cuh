// tmem.cuh -- tensor memory (tcgen05) helpers: allocation, 32-bit-per-lane loads and stores,
// and the tf32 MMA with operands in shared memory and the accumulator in tensor memory.
//
// Each SM has 512 columns x 128 lanes of 32-bit tensor memory.  A CTA of 4 warps allocates a
// power-of-two number of columns; warp w reads and writes lanes 32 w .. 32 w + 31 (lane =
// thread), so with the 32x32b shape every thread owns one lane: `.xN` moves N consecutive
// columns of it to or from N registers.  The allocation blocks while the SM has too few free
// columns, so a kernel that allocates C columns must never have more than 512 / C CTAs
// resident on an SM (the callers guarantee this by their shared-memory size).
#pragma once

#include <stdint.h>

#include "tma.cuh"

namespace ssm {

// One warp: allocates `ncols` columns and writes their base address to *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
// One warp: frees what tmem_alloc took.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Order tensor-memory operations around a thread barrier.
__device__ __forceinline__ void tmem_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Four columns of this thread's lane.
__device__ __forceinline__ void tmem_st4(uint32_t taddr, float a, float b, float c, float d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(__float_as_uint(c)),
               "r"(__float_as_uint(d))
               : "memory");
}
// Sixteen columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
// Waits until this thread's earlier stores have landed.
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Loads and waits in one statement, so the destination registers are never seen before the
// data is in them.
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
  uint32_t r0, r1, r2, r3;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(taddr)
      : "memory");
  v[0] = __uint_as_float(r0); v[1] = __uint_as_float(r1);
  v[2] = __uint_as_float(r2); v[3] = __uint_as_float(r3);
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

// Thirty-two columns of this thread's lane (load and wait in one statement).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

}  // namespace ssm

namespace ssm {
namespace tc {

// ---- tcgen05.mma, kind::tf32, operands in shared memory, accumulator in tensor memory -------
//
// Operand layout (the canonical K-major layout without swizzle): a tile of R rows x K columns of
// 32-bit elements is a grid of core matrices of 8 rows x 4 elements (8 x 16 bytes, stored as 128
// contiguous bytes, row r % 8 at 16 (r % 8) bytes); core matrix (row group r / 8, column group
// k / 4) starts at ((r / 8) (K / 4) + k / 4) 128 bytes.  The descriptor's leading byte offset is
// the step between core matrices along K (128 bytes), its stride byte offset the step between
// row groups (K / 4 x 128 bytes); one MMA of kind::tf32 consumes 8 columns (two core matrices
// along K), so consecutive K steps start 256 bytes apart.
//
// Accumulator rows in tensor memory: with M = 128, row r is lane r; with M = 64, row r is lane
// 32 (r / 16) + r % 16 (lanes 16..31 of every 32-lane group unused).

// Byte offset of the 16-byte row r % 8 of core matrix (r / 8, k4) in a K-major tile with K
// columns (k4 = k / 4).
__host__ __device__ __forceinline__ uint32_t kmajor_row16(uint32_t r, uint32_t k4, uint32_t K) {
  return ((r >> 3) * (K >> 2) + k4) * 128u + (r & 7u) * 16u;
}

// Shared-memory matrix descriptor of a K-major, unswizzled tile starting at `addr`.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t addr, uint32_t K) {
  const uint32_t lbo = 128u, sbo = (K >> 2) * 128u;
  uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version of sm_100-class devices
  return d;                // base offset 0, absolute leading offset, no swizzle
}

// Instruction descriptor: D fp32, A and B tf32, both K-major, shape M x N.
__host__ __device__ __forceinline__ constexpr uint32_t idesc_tf32(uint32_t M, uint32_t N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D (tensor memory) = A B^T (+ D when accumulate), one K step of 8 tf32 columns; one thread.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, bool accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}
// D (+)= A B^T over K columns of K-major tiles at a and b (shared-memory addresses).
__device__ __forceinline__ void mma_tf32_k(uint32_t d_tmem, uint32_t a, uint32_t b, uint32_t K,
                                           uint32_t idesc, bool accumulate) {
  for (uint32_t kk = 0; kk < K / 8; kk++)
    mma_tf32(d_tmem, desc_kmajor(a + kk * 256u, K), desc_kmajor(b + kk * 256u, K), idesc,
             accumulate || kk > 0);
}
// Arrives on the mbarrier once every MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// x rounded to the nearest tf32 value (10 explicit mantissa bits; low 13 bits zero).
__device__ __forceinline__ float tf32_rn(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

}  // namespace tc
}  // namespace ssm
